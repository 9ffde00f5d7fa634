// Causal per-document GQA attention backward on the tcgen05 tensor cores.
//
// Gradients of L with dL/dO = dO through the forward (SpecForge PR #728
// "feat(dspark): add Ulysses sequence parallel training", Accuracy Test:
// gradient parity with full-sequence attention):
//   P_tu  = exp(scale q_t.k_u - LSE_t),     delta_t = dO_t . O_t
//   dS_tu = P_tu (dO_t . v_u - delta_t)
//   dV_u  = sum_t P_tu dO_t,   dK_u = scale sum_t dS_tu q_t,
//   dQ_t  = scale sum_u dS_tu k_u.
//
// Three kernels, no atomics (so the result is deterministic):
//   delta_kernel  delta_t = dO_t . O_t                         (HBM-bound)
//   dkdv_kernel   one CTA per 128 key rows of one KV head; loops over the
//                 Hq/Hkv query heads of the group and the query tiles that
//                 see these keys, accumulating dV and dK in TMEM:
//                   S^T  = K Q^T,  dP^T = V dO^T        (SS MMA)
//                   P^T, dS^T computed per key row by 128 threads, both
//                   written as bf16 over S^T's TMEM region; S^T and dP^T
//                   swap regions every iteration
//                   dV  += P^T dO,  dK += dS^T Q        (TS MMA)
//   dq_kernel     one CTA per 128 query rows of one query head; loops over
//                 key tiles:  S = Q K^T, dP = dO V^T (SS), dS over S (bf16),
//                 dQ += dS K (TS).
// Both reuse the forward's warp roles: warp 0 TMA producer, warp 1 TMEM
// owner and MMA issuer (whole warp, one elected lane issues); warps 4-7 and 8-11 do the per-row elementwise work
// on the left and right 64 columns of each tile (two warps per SM
// sub-partition, so one hides the other's latency) and the epilogue.
// The bf16 values of each 32-column chunk are written over the first 16
// TMEM columns of that same chunk, so the two halves never touch each
// other's columns; the TS MMAs address K-step kk at column
// 32*(kk/2) + 8*(kk%2).  All waits are bounded (status word on timeout).
#include "tc_ptx.cuh"
#include "usp_common.cuh"

namespace {

using bf16 = __nv_bfloat16;
constexpr int BT = 128;                       // rows per tile (queries and keys)
// Twelve warps: 0 producer, 1 TMEM owner + MMA issuer, 2-3 idle, 4-11
// elementwise (warp % 4 is the TMEM lane quarter a warp may access).
constexpr int kThreads = 384;
constexpr int kEw0 = 4;                       // first elementwise warp
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory plan: NFIX stationary tiles, a ring of NS streamed tiles
// in NS/2 stages of two (one stage per iteration, one full and one empty
// barrier per stage), barriers, and (VEC) 128 fp32 staged next to each
// ring slot.
template <int D, int NFIX, int NS, bool VEC>
struct CfgT {
  static constexpr int NB = D / 64;
  static constexpr int BOX = 128 * 128;
  static constexpr int TILE = NB * BOX;
  static constexpr int NSTAGE = NS;
  static constexpr int NST2 = NS / 2;        // stages
  static_assert(NS % 2 == 0, "two tiles per stage");
  static constexpr int FIX_OFF = 0;
  static constexpr int RING_OFF = NFIX * TILE;
  static constexpr int BAR_OFF = RING_OFF + NSTAGE * TILE;
  static constexpr int VEC_OFF = BAR_OFF + 512;
  static constexpr int SMEM = VEC_OFF + (VEC ? NSTAGE * BT * 4 : 0) + 1024;
};
// dK/dV: K and V stationary, Q/dO streamed with LSE*log2(e)/delta vectors.
template <int D> using CfgKV = CfgT<D, 2, 4, true>;
// dQ: dO stationary (Q lives in TMEM), K/V streamed through six slots.
template <int D> using CfgQ = CfgT<D, 1, 6, false>;

struct Bars {
  uint64_t fix_full;
  uint64_t ring_full[4];   // per stage: both tiles (and vectors) landed
  uint64_t ring_empty[4];  // per stage: the MMAs reading it completed
  uint64_t sd_full;       // dq: S and dP of the iteration computed; dkdv: S^T computed
  uint64_t dp_full;       // dkdv: dP^T computed
  uint64_t consumed;      // dq: both elementwise groups read dP; dkdv: they read dP^T
                          // (256 arrivals)
  uint64_t s_consumed;    // dq: both elementwise groups read S (256 arrivals)
  uint64_t q_ready;       // dq: the Q tile is in TMEM (256 arrivals)
  uint64_t p_full[2];     // dkdv: P^T published ([0]), dS^T published ([1]);
                          // dq: dS written ([0]); 256 arrivals each
  uint64_t done[2];       // dkdv: dV MMA done ([0]), dK MMA done ([1]);
                          // dq: dQ MMA that read dS done ([0])
  uint64_t drain;         // wind-down: the MMAs issued so far completed
  uint32_t tmem_base;
  int abort;
};

struct Params {
  const int32_t* doc;
  const int32_t* cu;
  const bf16* q;         // head-layout Q (the dQ pass keeps its Q tile in TMEM)
  // both negated so that the elementwise code adds them with packed pair
  // instructions, which take no operand negation
  const float* nlse2;    // [P][hq][S_ws] -LSE*log2(e); -inf for rows without keys
  const float* ndelta;   // [P][hq][S_ws] -rowsum(dO*O); S_ws = S_pad rounded up to BT
  bf16* dq;
  bf16* dk;
  bf16* dv;
  int64_t S, S_pad, S_ws;
  int hq, hkv, G, n_tiles;
  int band_kv, band_q;   // head slots per band of the dkdv / dq CTA order (usp::cta_coords)
  int causal;            // 0: every key of a row's document is visible
  float scale, scale_log2;
  unsigned* status;
  int n_docs;              // entries of cu - 1 (index guards of debug builds)
  int64_t n_q, n_kv, n_ws; // elements of q/dq, of dk/dv, of each workspace vector
};

// Document of row t (-1 for a pad row); debug builds check the indices into
// doc and cu_seqlens and treat an out-of-range document id as a pad row.
__device__ __forceinline__ int doc_index(const Params& p, int64_t t) {
  if (t >= p.S || !usp::in_bounds(t, 1, p.S_pad, p.status)) return -1;
  const int d = __ldg(p.doc + t);
  if (d < 0 || (p.cu && !usp::in_bounds(d, 2, p.n_docs + 1, p.status))) return -1;
  return d;
}
__device__ __forceinline__ int64_t doc_start_of(const Params& p, int64_t t) {
  const int d = doc_index(p, t);
  if (d < 0) return -1;
  return p.cu ? (int64_t)__ldg(p.cu + d) : 0;
}
__device__ __forceinline__ int64_t doc_end_of(const Params& p, int64_t t) {
  const int d = doc_index(p, t);
  if (d < 0) return -1;
  return p.cu ? (int64_t)__ldg(p.cu + d + 1) : p.S;
}

// empty_count: commits that release a ring stage (one per issuing warp that
// reads it).
template <class C>
__device__ __forceinline__ void init_common(Bars* bars, int empty_count) {
  tc::mbar_init(&bars->fix_full, 1);
  for (int st = 0; st < C::NST2; ++st) {
    tc::mbar_init(&bars->ring_full[st], 1);
    tc::mbar_init(&bars->ring_empty[st], empty_count);
  }
  tc::mbar_init(&bars->sd_full, 1);
  tc::mbar_init(&bars->dp_full, 1);
  tc::mbar_init(&bars->consumed, 256);
  tc::mbar_init(&bars->s_consumed, 256);
  tc::mbar_init(&bars->q_ready, 256);
  for (int b = 0; b < 2; ++b) {
    tc::mbar_init(&bars->p_full[b], 256);
    tc::mbar_init(&bars->done[b], 1);
  }
  tc::mbar_init(&bars->drain, 1);
  bars->abort = 0;
  tc::fence_mbar_init();
}

// Producer: two stationary tiles (fixed coordinates) then `n_it` iterations
// of two streamed tiles each, one ring stage per iteration (slots 2st and
// 2st+1).  coord(it, w, c0, c1) gives the coordinates of streamed tile w of
// iteration it (map m0 or m1).  With VEC, vec(it, w) also names 128 fp32
// values copied next to the tile (into the slot's vector area; 512 bytes,
// 16-byte aligned).
template <class C, bool VEC, typename CoordFn, typename VecFn>
__device__ __forceinline__ void produce(uint8_t* smem, Bars* bars, volatile int* abort,
                                        const CUtensorMap* f0, int f0c0, const CUtensorMap* f1,
                                        int f1c0, int fc1, int g, const CUtensorMap* m0,
                                        const CUtensorMap* m1, int n_it, CoordFn coord,
                                        VecFn vec) {
  // f0 == nullptr: only f1 is loaded, into stationary tile 0
  const int nf = f0 != nullptr ? 2 : 1;
  tc::mbar_expect_tx(&bars->fix_full, nf * C::TILE);
  for (int b = 0; b < C::NB; ++b) {
    if (f0 != nullptr)
      tc::tma_load_3d(smem + C::FIX_OFF + b * C::BOX, f0, &bars->fix_full, f0c0 + b * 64, fc1, g);
    tc::tma_load_3d(smem + C::FIX_OFF + (nf - 1) * C::TILE + b * C::BOX, f1, &bars->fix_full,
                    f1c0 + b * 64, fc1, g);
  }
  int issued = 0;
  for (int it = 0; it < n_it && !*abort; ++it) {
    const int st = it % C::NST2, use = it / C::NST2;
    if (use > 0 && !tc::mbar_wait(&bars->ring_empty[st], (use - 1) & 1, abort)) break;
    tc::mbar_expect_tx(&bars->ring_full[st], 2 * (C::TILE + (VEC ? BT * 4 : 0)));
    for (int w = 0; w < 2; ++w) {
      const int s = 2 * st + w;
      int c0, c1;
      coord(it, w, c0, c1);
      for (int b = 0; b < C::NB; ++b)
        tc::tma_load_3d(smem + C::RING_OFF + s * C::TILE + b * C::BOX, w == 0 ? m0 : m1,
                        &bars->ring_full[st], c0 + b * 64, c1, g);
      if (VEC)
        tc::bulk_load(smem + C::VEC_OFF + s * BT * 4, vec(it, w), BT * 4, &bars->ring_full[st]);
    }
    ++issued;
  }
  if (*abort) {
    for (int it = (issued > C::NST2 ? issued - C::NST2 : 0); it < issued; ++it)
      tc::mbar_wait(&bars->ring_full[it % C::NST2], (it / C::NST2) & 1, nullptr, 100000000ull);
  }
}

// Issue T = F x R^T for one 128x128 tile pair (SS, K-major operands, K = D):
// F is a stationary tile, R a ring tile.
template <class C>
__device__ __forceinline__ void mma_tile_ss(uint32_t d_tmem, uint32_t f, uint32_t r) {
  constexpr int D = C::NB * 64;
  constexpr uint32_t id = tc::idesc_bf16(128, BT, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * C::BOX + (kk % 4) * 32;
    tc::mma_ss_w(d_tmem, tc::desc_sw128(f + off, 16, 1024), tc::desc_sw128(r + off, 16, 1024), id,
               kk > 0);
  }
}

// dK/dV MMA issuer.  Iteration `it` streams ring tiles Q (R0) and dO (R1).
// Two 128-column TMEM regions take turns: S^T(it) goes to region R (T0 for
// even it, T1 for odd) and dP^T(it) to the other region O.  The elementwise
// groups write P^T(it) as bf16 over the first 16 columns of each 32-column
// chunk of R and dS^T(it) over the other 16, so once they have read dP^T(it)
// out of O, O is free for S^T(it+1):
//   dV(it) += P^T(it) dO(it)   once P^T(it) is published   (TS, A from R)
//   S^T(it+1) = K Q^T  -> O    once dP^T(it) has been read (`consumed`)
//   dK(it) += dS^T(it) Q(it)   once dS^T(it) is published  (TS, A from R)
//   dP^T(it+1) = V dO^T -> R   once dK(it), and with it dV(it), completed
// S^T(it+1) thus waits for no MMA to finish, so the P^T phase of it+1 (the
// longer elementwise phase) runs while dK(it) and dP^T(it+1) execute; only
// dP^T(it+1) still waits for the pipe, since dK(it) reads R.
template <int D>
__device__ __forceinline__ void mma_loop_dkdv(uint8_t* smem, Bars* bars, volatile int* abort,
                                              uint32_t tmem, int n_it) {
  using C = CfgKV<D>;
  constexpr uint32_t A0 = 256, A1 = 256 + D;
  constexpr uint32_t id_acc = tc::idesc_bf16(128, D, true);
  const uint32_t fix = tc::smem_u32(smem + C::FIX_OFF);
  const uint32_t ring = tc::smem_u32(smem + C::RING_OFF);
  bool ok = tc::mbar_wait_warp(&bars->fix_full, 0, abort) &&
            tc::mbar_wait_warp(&bars->ring_full[0], 0, abort);
  if (ok) {
    tc::fence_after_sync();
    mma_tile_ss<C>(tmem + 0, fix, ring);
    tc::mma_commit_w(&bars->sd_full);
    mma_tile_ss<C>(tmem + 128, fix + C::TILE, ring + C::TILE);
    tc::mma_commit_w(&bars->dp_full);
  }
  for (int it = 0; ok && it < n_it; ++it) {
    const int st = it % C::NST2, nst = (it + 1) % C::NST2;
    const int s0 = 2 * st, s1 = 2 * st + 1, n0 = 2 * nst, n1 = 2 * nst + 1;
    const uint32_t R = (it & 1) ? 128u : 0u, O = 128u - R;
    const bool more = it + 1 < n_it;
    // dV(it) += P^T(it) dO(it)
    if (!(ok = tc::mbar_wait_warp(&bars->p_full[0], it & 1, abort))) break;
    tc::fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < BT / 16; ++kk)
      tc::mma_ts_w(tmem + A0, tmem + R + 32 * (kk >> 1) + 8 * (kk & 1),
                 tc::desc_sw128(ring + s1 * C::TILE + kk * 2048, C::BOX, 1024), id_acc,
                 (it > 0 || kk > 0) ? 1u : 0u);
    // S^T(it+1) into O once dP^T(it) has been read out of it
    if (more) {
      if (!(ok = tc::mbar_wait_warp(&bars->consumed, it & 1, abort))) break;
      if (!(ok = tc::mbar_wait_warp(&bars->ring_full[nst], ((it + 1) / C::NST2) & 1, abort))) break;
      tc::fence_after_sync();
      mma_tile_ss<C>(tmem + O, fix, ring + n0 * C::TILE);
      tc::mma_commit_w(&bars->sd_full);
    }
    // dK(it) += dS^T(it) Q(it)
    if (!(ok = tc::mbar_wait_warp(&bars->p_full[1], it & 1, abort))) break;
    tc::fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < BT / 16; ++kk)
      tc::mma_ts_w(tmem + A1, tmem + R + 16 + 32 * (kk >> 1) + 8 * (kk & 1),
                 tc::desc_sw128(ring + s0 * C::TILE + kk * 2048, C::BOX, 1024), id_acc,
                 (it > 0 || kk > 0) ? 1u : 0u);
    tc::mma_commit_w(&bars->done[1]);
    tc::mma_commit_w(&bars->ring_empty[st]);
    // dP^T(it+1) into R once dV(it) and dK(it) have read P^T(it), dS^T(it)
    if (more) {
      if (!(ok = tc::mbar_wait_warp(&bars->done[1], it & 1, abort))) break;
      tc::fence_after_sync();
      mma_tile_ss<C>(tmem + R, fix + C::TILE, ring + n1 * C::TILE);
      tc::mma_commit_w(&bars->dp_full);
    }
  }
  if (!ok) {
    tc::mma_commit_w(&bars->drain);
    tc::mbar_wait(&bars->drain, 0, nullptr, 100000000ull);
  }
}

// dQ MMA issuer.  The Q tile of this CTA sits in TMEM (columns QC..QC+63,
// written once by the elementwise groups), so S needs no shared-memory
// reads for its A operand.  Iteration j streams key tile K_j and V_j (one
// ring stage):
//   S(j) = Q K_j^T (T0, TS),  dP(j) = dO V_j^T (T1, SS)
//   dQ += dS(j) K_j   with dS(j) in TMEM columns R..R+63              (TS)
// S(j+1) is issued as soon as the elementwise groups have read S(j)
// (`s_consumed`) and dP(j+1) as soon as they have read dP(j) (`consumed`),
// before they finish dS(j), so the tensor pipe keeps working while they
// read dP and compute.  The dS columns are rewritten for j+1
// only after done[0] of dQ(j).  (Issuing dQ from a second warp was slower:
// the two streams interleave their MMAs in the pipe.)
template <int D>
__device__ __forceinline__ void mma_tile_s_ts(uint32_t d_tmem, uint32_t q_tmem, uint32_t k) {
  using C = CfgQ<D>;
  constexpr uint32_t id = tc::idesc_bf16(128, BT, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * C::BOX + (kk % 4) * 32;
    tc::mma_ts_w(d_tmem, q_tmem + 8 * kk, tc::desc_sw128(k + off, 16, 1024), id, kk > 0);
  }
}

// dQ kernel TMEM columns: S, dP, the dQ accumulator, dS (bf16), Q (bf16)
constexpr uint32_t kDqT0 = 0, kDqT1 = 128, kDqAcc = 256, kDqR = 384, kDqQ = 448;

template <int D>
__device__ __forceinline__ void mma_loop_dq(uint8_t* smem, Bars* bars, volatile int* abort,
                                            uint32_t tmem, int n_it) {
  using C = CfgQ<D>;
  constexpr uint32_t id_acc = tc::idesc_bf16(128, D, true);
  const uint32_t fix = tc::smem_u32(smem + C::FIX_OFF);
  const uint32_t ring = tc::smem_u32(smem + C::RING_OFF);
  bool ok = tc::mbar_wait_warp(&bars->fix_full, 0, abort) &&
            tc::mbar_wait_warp(&bars->q_ready, 0, abort) &&
            tc::mbar_wait_warp(&bars->ring_full[0], 0, abort);
  if (ok) {
    tc::fence_after_sync();
    mma_tile_s_ts<D>(tmem + kDqT0, tmem + kDqQ, ring);
    mma_tile_ss<C>(tmem + kDqT1, fix, ring + C::TILE);
    tc::mma_commit_w(&bars->sd_full);
  }
  for (int j = 0; ok && j < n_it; ++j) {
    const int st = j % C::NST2, s0 = 2 * st;
    if (j + 1 < n_it) {
      const int nst = (j + 1) % C::NST2, n0 = 2 * nst, n1 = 2 * nst + 1;
      if (!(ok = tc::mbar_wait_warp(&bars->s_consumed, j & 1, abort))) break;
      if (!(ok = tc::mbar_wait_warp(&bars->ring_full[nst], ((j + 1) / C::NST2) & 1, abort))) break;
      tc::fence_after_sync();
      mma_tile_s_ts<D>(tmem + kDqT0, tmem + kDqQ, ring + n0 * C::TILE);
      if (!(ok = tc::mbar_wait_warp(&bars->consumed, j & 1, abort))) break;
      tc::fence_after_sync();
      mma_tile_ss<C>(tmem + kDqT1, fix, ring + n1 * C::TILE);
      tc::mma_commit_w(&bars->sd_full);
    }
    if (!(ok = tc::mbar_wait_warp(&bars->p_full[0], j & 1, abort))) break;
    tc::fence_after_sync();
#pragma unroll
    for (int kk = 0; kk < BT / 16; ++kk)
      tc::mma_ts_w(tmem + kDqAcc, tmem + kDqR + 8 * kk,
                   tc::desc_sw128(ring + s0 * C::TILE + kk * 2048, C::BOX, 1024), id_acc,
                   (j > 0 || kk > 0) ? 1u : 0u);
    tc::mma_commit_w(&bars->done[0]);
    tc::mma_commit_w(&bars->ring_empty[st]);     // K_j (S(j), dQ(j)) and V_j (dP(j))
  }
  if (!ok) {
    tc::mma_commit_w(&bars->drain);
    tc::mbar_wait(&bars->drain, 0, nullptr, 100000000ull);
  }
}

// dK/dV elementwise work on half h (queries [64h, 64h+64)) of this thread's
// key row, in two phases so that each overlaps an MMA:
//   phase 1: P^T = exp2(S^T*sl2 - lse2[col]) from region R, written as bf16
//            over R (first 16 columns of each 32-column chunk) and kept, as
//            the same bf16 pairs, in 32 registers;
//   phase 2: dS^T = P^T (dP^T - delta[col]) with dP^T read from region O
//            (which the thread then reports `consumed`), written as bf16
//            over R (last 16 columns of each chunk).
// dS^T is thus formed from the bf16 P^T that dV is built from (a relative
// change of at most 2^-9 per element, the size of the rounding dS^T gets
// anyway).  The per-column lse2 and delta come in registers, negated (the
// workspace stores -lse2 and -delta), and pairs of columns go through packed
// fp32x2 instructions.
// bf16 values of each 32-column chunk go to that chunk's first 16 columns.
// Columns outside [lo, hi] are zero when MASK.
template <bool MASK>
__device__ __forceinline__ void dkdv_phase_p(uint32_t tS, int h, int lo, int hi,
                                             const float (&l2)[64], float sl2, uint32_t (&pk)[32]) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {   // two 32-column chunks (fewer live registers)
    uint32_t sv[32];
    tc::tmem_ld_x32(tS + 64 * h + 32 * cc, sv);
    uint32_t pw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {   // pairs of columns: one packed fma per pair
      float pv[2];
      const int k = 32 * cc + 2 * i;
      tc::fma2(pv[0], pv[1], __uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]), sl2,
               sl2, l2[k], l2[k + 1]);   // l2 holds -LSE*log2(e)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        pv[e] = tc::ex2(pv[e]);
        if (MASK) {
          const int col = 64 * h + k + e;
          if (!(col >= lo && col <= hi)) pv[e] = 0.f;
        }
      }
      pw[i] = tc::pack_bf16(pv[0], pv[1]);
      pk[16 * cc + i] = pw[i];
    }
    tc::tmem_st_x16(tS + 64 * h + 32 * cc, pw);
  }
}

__device__ __forceinline__ void dkdv_phase_ds(uint32_t tP, uint32_t tS, int h,
                                              const float (&d2)[64], const uint32_t (&pk)[32],
                                              Bars* bars) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t dv[32];
    tc::tmem_ld_x32(tP + 64 * h + 32 * cc, dv);
    if (cc == 1) {          // all of this thread's dP^T columns are read
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->consumed);
    }
    uint32_t dw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w = pk[16 * cc + i];
      const float p0 = __uint_as_float(w << 16), p1 = __uint_as_float(w & 0xffff0000u);
      const int k = 32 * cc + 2 * i;
      float t0, t1;   // (dP^T - delta) P^T with d2 holding -delta, as packed pairs
      tc::add2(t0, t1, __uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1]), d2[k],
               d2[k + 1]);
      tc::mul2(t0, t1, p0, p1, t0, t1);
      dw[i] = tc::pack_bf16(t0, t1);
    }
    tc::tmem_st_x16(tS + 64 * h + 32 * cc + 16, dw);
  }
}

// 64 fp32 values from shared memory (the same address in every lane) into
// registers.  The loads are issued early, where the warp would wait anyway:
// while the SS MMAs stream their operands, a shared-memory load issued in
// the middle of an elementwise phase waits a long time for its turn.
__device__ __forceinline__ void load_vec64(const float* src, float (&v)[64]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 a = reinterpret_cast<const float4*>(src)[i];
    v[4 * i] = a.x; v[4 * i + 1] = a.y; v[4 * i + 2] = a.z; v[4 * i + 3] = a.w;
  }
}

// dQ elementwise work on half h (keys [64h, 64h+64)) of this thread's query
// row: read S and dP, let the MMA issuer reuse them ("consumed"), compute
// dS = exp2(S*sl2 - lse2) (dP - delta) (with nlse2 = -lse2 and ndl = -delta,
// as packed pairs) and, once the dS columns are free,
// write it there as bf16 (32 columns: K steps 4h..4h+3).
template <bool MASK>
__device__ __forceinline__ bool dq_half(uint32_t tS, uint32_t tP, uint32_t tR, int h, int lo,
                                        int hi, float nlse2, float ndl, float sl2, Bars* bars,
                                        int j, volatile int* abort) {
  uint32_t sv[64], dv[64];
  tc::tmem_ld_x64(tS + 64 * h, sv);
  tc::fence_before_sync();
  tc::mbar_arrive(&bars->s_consumed);      // S(j+1) may overwrite S now
  tc::tmem_ld_x64(tP + 64 * h, dv);
  tc::fence_before_sync();
  tc::mbar_arrive(&bars->consumed);
  uint32_t w[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float x0, x1, t0, t1;
    tc::fma2(x0, x1, __uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]), sl2, sl2, nlse2,
             nlse2);
    tc::add2(t0, t1, __uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1]), ndl, ndl);
    float dd[2];
    tc::mul2(dd[0], dd[1], tc::ex2(x0), tc::ex2(x1), t0, t1);
    if (MASK) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = 64 * h + 2 * i + e;
        if (!(col >= lo && col <= hi)) dd[e] = 0.f;
      }
    }
    w[i] = tc::pack_bf16(dd[0], dd[1]);
  }
  if (j >= 1) {   // the dQ MMA of iteration j-1 read the dS columns
    if (!tc::mbar_wait_warp(&bars->done[0], (j - 1) & 1, abort))
      return false;
    tc::fence_after_sync();
  }
  tc::tmem_st_x32(tR + 32 * h, w);
  return true;
}

// Store 32 fp32 values (times f) of one row as bf16 to global.
__device__ __forceinline__ void store_row32(bf16* dst, const uint32_t (&v)[32], float f) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    w[i] = tc::pack_bf16(__uint_as_float(v[2 * i]) * f, __uint_as_float(v[2 * i + 1]) * f);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// ------------------------------------------------------------------- dK, dV
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const Params p) {
  using C = CfgKV<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFF);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // rank 0 = key tile 0, which every causal query sees (the heaviest)
  int rank, y;
  usp::cta_coords(p.n_tiles, p.band_kv, rank, y);
  const int64_t u0 = (int64_t)rank * BT;
  const int g = y / p.hkv;
  const int jk = y % p.hkv;
  // query rows that see these keys: from u0 (causal) or the first key's
  // document start, to the end of the last valid key's document
  int n_q = 0;
  int64_t tq0 = 0;
  {
    const int64_t last = min(u0 + BT, p.S) - 1;
    if (last >= u0) {
      const int64_t e = doc_end_of(p, last);
      tq0 = ((p.causal ? u0 : doc_start_of(p, u0)) / BT) * BT;
      n_q = (int)((e - tq0 + BT - 1) / BT);
    }
  }
  const int n_it = n_q * p.G;    // iteration it: query tile it / G, head jk*G + it % G

  if (threadIdx.x == 0) init_common<C>(bars, 1);
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    if (lane == 0 && n_it > 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmdO);
      const int G = p.G;
      produce<C, true>(
          smem, bars, abort, &tmK, jk * D, &tmV, jk * D, (int)u0, g, &tmQ, &tmdO, n_it,
          [&](int it, int, int& c0, int& c1) {
            c0 = (jk * G + it % G) * D;
            c1 = (int)(tq0 + (int64_t)(it / G) * BT);
          },
          [&](int it, int w) -> const float* {
            // lse2 next to the Q tile, delta next to the dO tile
            const int64_t off = ((int64_t)g * p.hq + jk * G + it % G) * p.S_ws + tq0 +
                                (int64_t)(it / G) * BT;
            // debug builds: an out-of-range vector is reported and replaced
            // by the first one, so that the copy still completes its barrier
            const bool in = usp::in_bounds(off, BT, p.n_ws, p.status);
            return (w == 0 ? p.nlse2 : p.ndelta) + (in ? off : 0);
          });
    }
  } else if (warp == 1) {
    if (n_it > 0) mma_loop_dkdv<D>(smem, bars, abort, tmem, n_it);   // whole warp
  } else if (warp >= kEw0) {
    const int quarter = warp & 3;
    const int half = (warp - kEw0) >> 2;       // columns [64*half, 64*half + 64)
    const int r = quarter * 32 + lane;
    const int64_t u = u0 + r;
    const int64_t de = doc_end_of(p, u);         // queries [qs, de) see key u
    const int64_t qs = p.causal ? u : doc_start_of(p, u);
    // the two TMEM regions that S^T and dP^T alternate between
    const uint32_t tT0 = tc::tmem_addr(tmem, quarter * 32, 0);
    const uint32_t tT1 = tc::tmem_addr(tmem, quarter * 32, 128);
    // per-query LSE*log2(e) (next to the Q tile) and delta (next to the dO
    // tile) of this half's 64 columns, staged by the producer
    const float* vec = reinterpret_cast<const float*>(smem + C::VEC_OFF) + 64 * half;
    float l2[64];
    bool ok = true;
    if (n_it > 0) {
      ok = tc::mbar_wait_warp(&bars->ring_full[0], 0, abort);
      if (ok) load_vec64(vec, l2);
    }
    for (int it = 0; ok && it < n_it; ++it) {
      const int64_t t0 = tq0 + (int64_t)(it / p.G) * BT;
      const int s1 = 2 * (it % C::NST2) + 1;     // this stage's dO slot (delta)
      const uint32_t tS = (it & 1) ? tT1 : tT0;  // S^T(it), then P^T, dS^T
      const uint32_t tP = (it & 1) ? tT0 : tT1;  // dP^T(it)
      ok = tc::mbar_wait_warp(&bars->sd_full, it & 1, abort);
      if (!ok) break;
      tc::fence_after_sync();
      const int lo = (int)max((int64_t)0, min((int64_t)BT, qs - t0));
      const int hi = de < 0 ? -1 : (int)min((int64_t)BT - 1, de - 1 - t0);
      const bool mask = __any_sync(0xffffffffu, lo > 64 * half || hi < 64 * half + 63);
      uint32_t pk[32];
      if (mask) dkdv_phase_p<true>(tS, half, lo, hi, l2, p.scale_log2, pk);
      else dkdv_phase_p<false>(tS, half, lo, hi, l2, p.scale_log2, pk);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->p_full[0]);
      float d2[64];
      load_vec64(vec + s1 * BT, d2);
      ok = tc::mbar_wait_warp(&bars->dp_full, it & 1, abort);
      if (!ok) break;
      tc::fence_after_sync();
      dkdv_phase_ds(tP, tS, half, d2, pk, bars);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->p_full[1]);
      // the next iteration's lse2, loaded while the S^T MMA runs (after the
      // last iteration the loads read a slot's stale values, never used: an
      // unconditional load keeps the old values from living through phase 2)
      const int nst = (it + 1) % C::NST2;
      if (it + 1 < n_it)
        ok = tc::mbar_wait_warp(&bars->ring_full[nst], ((it + 1) / C::NST2) & 1, abort);
      load_vec64(vec + 2 * nst * BT, l2);
    }
    if (ok && n_it > 0) {   // dK is the last MMA; it completes after dV
      ok = tc::mbar_wait_warp(&bars->done[1], (n_it - 1) & 1, abort);
      tc::fence_after_sync();
    }
    // epilogue: the left half writes dV, the right half dK
    const bool have = ok && n_it > 0;          // warp-uniform
    const int64_t row_off = (((int64_t)g * p.S_pad + u) * p.hkv + jk) * D;
    bf16* row = (half == 0 ? p.dv : p.dk) + row_off;
    const uint32_t acc = 256 + half * D;
    const float f = half == 0 ? 1.f : p.scale;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t v[32];
      if (have) {
        tc::tmem_ld_x32(tc::tmem_addr(tmem, quarter * 32, acc + c * 32), v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      if (u < p.S_pad && usp::in_bounds(row_off + c * 32, 32, p.n_kv, p.status))
        store_row32(row + c * 32, v, f);
    }
  }
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  if (*abort && threadIdx.x == 0) usp::set_status(p.status, usp::kErrTimeout);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------- dQ
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const Params p) {
  using C = CfgQ<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFF);
  volatile int* abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // rank 0 = the last query tile, the heaviest causal one
  int rank, y;
  usp::cta_coords(p.n_tiles, p.band_q, rank, y);
  const int qt = p.n_tiles - 1 - rank;
  const int64_t t0 = (int64_t)qt * BT;
  const int g = y / p.hq;
  const int jq = y % p.hq;
  const int jk = jq / p.G;
  int n_kv = 0;
  int64_t kv_start = 0;
  {
    const int64_t ds0 = doc_start_of(p, t0);
    if (ds0 >= 0) {
      kv_start = (ds0 / BT) * BT;
      const int64_t last = min(t0 + BT, p.S) - 1;
      const int64_t kv_end = p.causal ? last + 1 : doc_end_of(p, last);
      n_kv = (int)((kv_end - kv_start + BT - 1) / BT);
    }
  }

  if (threadIdx.x == 0) init_common<C>(bars, 1);
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    if (lane == 0 && n_kv > 0) {
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      produce<C, false>(
          smem, bars, abort, nullptr, 0, &tmdO, jq * D, (int)t0, g, &tmK, &tmV, n_kv,
          [&](int it, int, int& c0, int& c1) {
            c0 = jk * D;
            c1 = (int)(kv_start + (int64_t)it * BT);
          },
          [&](int, int) -> const float* { return nullptr; });
    }
  } else if (warp == 1) {
    if (n_kv > 0) mma_loop_dq<D>(smem, bars, abort, tmem, n_kv);     // whole warp
  } else if (warp >= kEw0) {
    const int quarter = warp & 3;
    const int half = (warp - kEw0) >> 2;       // columns [64*half, 64*half + 64)
    const int r = quarter * 32 + lane;
    const int64_t t = t0 + r;
    const int64_t ds = doc_start_of(p, t);
    // last key row t sees: itself (causal) or its document's last row
    const int64_t ke = ds < 0 ? -1 : (p.causal ? t : doc_end_of(p, t) - 1);
    float nlse2 = -INFINITY, ndl = 0.f;
    if (ds >= 0) {
      const int64_t li = ((int64_t)g * p.hq + jq) * p.S_ws + t;
      if (usp::in_bounds(li, 1, p.n_ws, p.status)) {
        nlse2 = __ldg(p.nlse2 + li);
        ndl = __ldg(p.ndelta + li);
      }
    }
    const uint32_t tS = tc::tmem_addr(tmem, quarter * 32, kDqT0);
    const uint32_t tP = tc::tmem_addr(tmem, quarter * 32, kDqT1);
    bool ok = true;
    // this thread's Q row, columns [64*half, 64*half + 64), into TMEM as
    // the A operand of S = Q K^T (bf16 pairs, 32 columns)
    {
      uint32_t qw[32];
      const bool mine = D == 128 || half == 0;     // D = 64: the left group holds the row
      const int64_t q_off = (((int64_t)g * p.S_pad + t) * p.hq + jq) * D + (mine ? 64 * half : 0);
      const uint4* src = reinterpret_cast<const uint4*>(p.q + q_off);
      const bool rd = t < p.S_pad && mine && usp::in_bounds(q_off, 64, p.n_q, p.status);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = rd ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        qw[4 * i] = v.x; qw[4 * i + 1] = v.y; qw[4 * i + 2] = v.z; qw[4 * i + 3] = v.w;
      }
      if (D == 128 || half == 0)
        tc::tmem_st_x32(tc::tmem_addr(tmem, quarter * 32, kDqQ + 32 * half), qw);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->q_ready);
    }
    const uint32_t tR = tc::tmem_addr(tmem, quarter * 32, kDqR);
    for (int it = 0; it < n_kv; ++it) {
      ok = tc::mbar_wait_warp(&bars->sd_full, it & 1, abort);
      if (!ok) break;
      tc::fence_after_sync();
      const int64_t u0 = kv_start + (int64_t)it * BT;
      const int lo = (int)max((int64_t)0, min((int64_t)BT, ds - u0));
      const int hi = ds < 0 ? -1 : (int)max((int64_t)-1, min((int64_t)BT - 1, ke - u0));
      const bool mask = __any_sync(0xffffffffu, lo > 64 * half || hi < 64 * half + 63);
      const uint32_t tRb = tR;
      ok = mask ? dq_half<true>(tS, tP, tRb, half, lo, hi, nlse2, ndl, p.scale_log2, bars, it,
                                abort)
                : dq_half<false>(tS, tP, tRb, half, lo, hi, nlse2, ndl, p.scale_log2, bars, it,
                                 abort);
      if (!ok) break;
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&bars->p_full[0]);
    }
    if (ok && n_kv > 0) {   // the last dQ MMA completes after all earlier ones
      ok = tc::mbar_wait_warp(&bars->done[0], (n_kv - 1) & 1, abort);
      tc::fence_after_sync();
    }
    const bool have = ok && n_kv > 0;
    const int64_t row_off = (((int64_t)g * p.S_pad + t) * p.hq + jq) * D;
    bf16* row = p.dq + row_off;
#pragma unroll
    for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
      uint32_t v[32];
      if (have) {
        tc::tmem_ld_x32(tc::tmem_addr(tmem, quarter * 32, kDqAcc + c * 32), v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      if (t < p.S_pad && usp::in_bounds(row_off + c * 32, 32, p.n_q, p.status))
        store_row32(row + c * 32, v, ds >= 0 ? p.scale : 0.f);
    }
  }
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  if (*abort && threadIdx.x == 0) usp::set_status(p.status, usp::kErrTimeout);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------ delta = rowsum(dO*O)
// D/8 lanes per (row, head): 16-byte loads, fp32 products and a shuffle sum;
// a warp takes 32/(D/8) rows at a time, four such groups per step.
// Writes both negated: ndelta = -delta and nlse2 = -LSE*log2(e) (-inf where
// LSE = -inf).  Both arrays have rows of S_ws >= S_pad entries; entries
// [S_pad, S_ws) get ndelta 0 and nlse2 -inf.
template <int D>
__global__ void __launch_bounds__(256) delta_kernel(const bf16* __restrict__ o,
                                                    const bf16* __restrict__ dout,
                                                    const float* __restrict__ lse,
                                                    float* __restrict__ delta,
                                                    float* __restrict__ lse2, int64_t S_pad,
                                                    int64_t S_ws, int hq, int64_t n_rows,
                                                    unsigned* status) {
  const int64_t n_ws = (n_rows / S_pad) * S_ws;    // entries of each workspace vector
  {
    const int64_t extra = S_ws - S_pad;
    const int64_t n_extra = (n_rows / S_pad) * extra;     // (P*hq) rows
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_extra;
         i += (int64_t)gridDim.x * blockDim.x) {
      const int64_t rr = i / extra;
      const int64_t idx = rr * S_ws + S_pad + (i - rr * extra);
      if (!usp::in_bounds(idx, 1, n_ws, status)) continue;
      delta[idx] = 0.f;
      lse2[idx] = -INFINITY;
    }
  }
  constexpr int LPR = D / 8;                  // lanes per row (8 bf16 each)
  constexpr int RPW = 32 / LPR;               // rows per warp step
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // U row groups per warp step: the loads of all of them are issued before
  // any is used, so each lane keeps 2*U 16-byte loads in flight
  constexpr int U = 4;
  for (int64_t base = w0 * RPW * U; base < n_rows; base += nw * RPW * U) {
    uint4 a[U], b[U];
    int64_t row[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      row[u] = base + u * RPW + lane / LPR;   // row = (g*S_pad + t)*hq + j
      ok[u] = row[u] < n_rows &&
              usp::in_bounds(row[u] * D + 8 * (lane % LPR), 8, n_rows * D, status);
      a[u] = ok[u] ? __ldcs(reinterpret_cast<const uint4*>(o + row[u] * D) + lane % LPR)
                   : make_uint4(0, 0, 0, 0);
      b[u] = ok[u] ? __ldcs(reinterpret_cast<const uint4*>(dout + row[u] * D) + lane % LPR)
                   : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float s = 0.f;
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b[u]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 fa = __bfloat1622float2(pa[i]);
        const float2 fb = __bfloat1622float2(pb[i]);
        s = fmaf(fa.x, fb.x, s);
        s = fmaf(fa.y, fb.y, s);
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (row[u] < n_rows && lane % LPR == 0) {
        const int64_t gt = row[u] / hq;
        const int j = (int)(row[u] - gt * hq);
        const int64_t g = gt / S_pad, t = gt - g * S_pad;
        const int64_t li = (g * hq + j) * S_ws + t;
        const int64_t lj = (g * hq + j) * S_pad + t;
        if (usp::in_bounds(li, 1, n_ws, status) && usp::in_bounds(lj, 1, n_rows, status)) {
          delta[li] = -s;
          const float x = lse[lj];
          lse2[li] = x == -INFINITY ? -INFINITY : -(x * kLog2e);
        }
      }
    }
  }
}

template <int D>
cudaError_t launch_all(const usp::Geometry& g, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, const Params& prm,
                       const bf16* o, const bf16* dout, const float* lse, float* delta,
                       float* lse2, cudaStream_t st) {
  const int64_t n_kv_cta = (int64_t)prm.n_tiles * g.P * g.hkv;
  const int64_t n_q_cta = (int64_t)prm.n_tiles * g.P * g.hq;
  if (n_q_cta > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const int64_t n_rows = (int64_t)g.P * g.S_pad * g.hq;
  int64_t blocks = (n_rows * (D / 8) * 1 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  delta_kernel<D><<<(int)(blocks < 1 ? 1 : blocks), 256, 0, st>>>(
      o, dout, lse, delta, lse2, g.S_pad, prm.S_ws, g.hq, n_rows, prm.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int smem_kv = CfgKV<D>::SMEM, smem_q = CfgQ<D>::SMEM;
  static_assert(smem_kv <= 232448 && smem_q <= 232448, "shared memory plan too large");
  if ((e = cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_kv)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_q)) != cudaSuccess)
    return e;
  dkdv_kernel<D><<<(unsigned)n_kv_cta, kThreads, smem_kv, st>>>(mq, mk, mv, mdo, prm);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dq_kernel<D><<<(unsigned)n_q_cta, kThreads, smem_q, st>>>(mq, mk, mv, mdo, prm);
  usp_count_launches(3);
  return cudaGetLastError();
}

}  // namespace

// Workspace: delta and lse2, each [P][hq][S_ws] fp32 with S_ws = S_pad
// rounded up to a multiple of BT.  Sizes that do not fit in size_t give
// SIZE_MAX, which no workspace (and no fixed scratch) satisfies.
static int64_t ws_row(const usp::Geometry& g) { return (g.S_pad + BT - 1) / BT * BT; }
static size_t vec_bytes(const usp::Geometry& g) {
  const uint64_t rows = (uint64_t)g.P * (uint64_t)g.hq;
  const uint64_t row_bytes = (uint64_t)ws_row(g) * sizeof(float);
  const uint64_t cap = (SIZE_MAX / 2 - 255);
  if (row_bytes != 0 && rows > cap / row_bytes) return SIZE_MAX;
  const size_t n = (size_t)(rows * row_bytes);
  return ((n + 255) / 256) * 256;
}
size_t usp_attn_bwd_ws_bytes(const usp::Geometry& g) {
  const size_t v = vec_bytes(g);
  return v == SIZE_MAX ? SIZE_MAX : 2 * v;
}

cudaError_t usp_launch_attn_bwd(const usp::Geometry& g, const void* q, const void* k,
                                const void* v, const void* o, const float* lse,
                                const void* dout, const int32_t* doc, const int32_t* cu,
                                void* dq, void* dk, void* dv, void* ws, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdo;
  if (!usp_make_head_map(&mq, q, g.hq, g.D, g.S_pad, g.P, 128) ||
      !usp_make_head_map(&mk, k, g.hkv, g.D, g.S_pad, g.P, 128) ||
      !usp_make_head_map(&mv, v, g.hkv, g.D, g.S_pad, g.P, 128) ||
      !usp_make_head_map(&mdo, dout, g.hq, g.D, g.S_pad, g.P, 128))
    return cudaErrorInvalidValue;
  Params prm;
  prm.doc = doc;
  prm.cu = cu;
  prm.q = reinterpret_cast<const bf16*>(q);
  float* delta = reinterpret_cast<float*>(ws);
  float* lse2 = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + vec_bytes(g));
  prm.nlse2 = lse2;
  prm.ndelta = delta;
  prm.dq = reinterpret_cast<bf16*>(dq);
  prm.dk = reinterpret_cast<bf16*>(dk);
  prm.dv = reinterpret_cast<bf16*>(dv);
  prm.S = g.S;
  prm.S_pad = g.S_pad;
  prm.S_ws = ws_row(g);
  prm.hq = g.hq;
  prm.hkv = g.hkv;
  prm.G = g.G;
  prm.causal = g.causal;
  prm.n_tiles = (int)((g.S_pad + BT - 1) / BT);
  prm.band_kv = usp::cta_band(prm.n_tiles, g.P * g.hkv);
  prm.band_q = usp::cta_band(prm.n_tiles, g.P * g.hq);
  prm.scale = g.scale;
  prm.scale_log2 = g.scale * kLog2e;
  prm.status = g.status;
  prm.n_docs = g.n_docs;
  prm.n_q = (int64_t)g.P * g.S_pad * g.hq * g.D;
  prm.n_kv = (int64_t)g.P * g.S_pad * g.hkv * g.D;
  prm.n_ws = (int64_t)g.P * g.hq * prm.S_ws;
  const bf16* ob = reinterpret_cast<const bf16*>(o);
  const bf16* db = reinterpret_cast<const bf16*>(dout);
  if (g.D == 128) return launch_all<128>(g, mq, mk, mv, mdo, prm, ob, db, lse, delta, lse2, st);
  return launch_all<64>(g, mq, mk, mv, mdo, prm, ob, db, lse, delta, lse2, st);
}

// ---------------------------------------------------------------------------
// Fixed scratch for usp_attn_bwd_noalloc: callers that cannot allocate device
// memory get the backward's workspace (delta and LSE*log2(e)) from this array
// instead.  Every GPU that loads the library holds it until the process
// exits.  All calls share it and it keeps the last call's contents; the
// backward rewrites every entry it reads, so nothing has to be cleared
// between calls, but calls that overlap on the GPU race on it.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

size_t usp_noalloc_scratch_capacity() { return kNoAllocScratchBytes; }

// Device address of the scratch array on the current device, looked up
// with that device current on every call: the first lookup on a device
// loads this module there (under lazy loading) and with it the array; later
// lookups are a table read.  Nothing is cached, so concurrent first calls
// from several host threads do not race and no address outlives its
// context.
cudaError_t usp_noalloc_scratch(void** ptr) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *ptr = p;
  return cudaSuccess;
}
