// Causal per-document GQA attention forward on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), sm_103a.
//
// What it computes (SpecForge PR #728 "feat(dspark): add Ulysses sequence
// parallel training", Modifications: local attention of each rank's head
// group after the all-to-all; Accuracy Test: equal to full-sequence
// attention): for every head group g, query head j and row t
//   O[t] = sum_{u in M(t)} softmax_u(scale q_t.k_u) v_u,  LSE[t] = ln sum exp(..)
// with M(t) = {u : doc(u) == doc(t) >= 0, u <= t}.
//
// Design (one CTA = 128 query rows x NH query heads that share one KV head):
//   warp 0      TMA producer: Q tiles once, then K/V tiles through an
//               NSTAGE-deep shared-memory ring (128-byte swizzle).
//   warp 1      TMEM allocation and MMA issue (the whole warp runs the
//               loop, one elected lane issues each instruction):
//               S_h = Q_h K^T (SS MMA, 128x128x D) into TMEM,
//               O_h += P_h V   (TS MMA: P read from TMEM, V from smem).
//   warps 4-7   softmax of head slot 0, warps 8-11 of slot 1: one thread
//               per query row reads its S row from TMEM, applies the mask,
//               runs the online softmax in the exp2 domain, writes P (bf16)
//               back over S, rescales its O row in TMEM only when its
//               running max grew by more than 2^8, and finally normalises
//               O and writes O (bf16) and LSE.
// Sharing K/V between the NH heads of a GQA group halves K/V shared-memory
// traffic, and the two heads' MMA chains interleave so that one head's
// softmax overlaps the other head's MMAs.  Every wait is bounded: on a
// timeout the CTA records it in the status word and winds down.
#include "tc_ptx.cuh"
#include "usp_common.cuh"

#include <cudaTypedefs.h>

namespace {

using bf16 = __nv_bfloat16;
constexpr int BM = 128;   // query rows per tile
constexpr int BN = 128;   // key rows per tile
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D, int NH>
struct Cfg {
  static constexpr int NB = D / 64;                  // 128-byte column boxes per tile
  static constexpr int BOX = 128 * 128;              // bytes of one [128 rows][64 cols] box
  static constexpr int TILE = NB * BOX;              // one 128-row tile of D columns
  static constexpr int NSTAGE = D == 128 ? 4 : 6;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = NH * TILE;
  static constexpr int BAR_OFF = KV_OFF + NSTAGE * TILE;
  static constexpr int SMEM = BAR_OFF + 512 + 1024;   // barriers + alignment slack
  static_assert(SMEM <= 232448, "shared memory plan too large");
  // TMEM columns: S/P of slot h at h*128, O of slot h at 256 + h*D
  static constexpr uint32_t S_COL(int h) { return h * 128; }
  static constexpr uint32_t O_COL(int h) { return 256 + h * D; }
};

struct Params {
  const int32_t* doc;
  const int32_t* cu;
  bf16* o;
  float* lse;
  int64_t S, S_pad;
  int hq, hkv, G, n_qtiles, slots_per_kv;
  int band;               // head slots per band of the CTA order (usp::cta_coords)
  int causal;             // 0: every key of the row's document is visible
  int64_t k_lo, k_hi;     // key window: only rows [k_lo, k_hi) are keys
  float scale_log2;
  unsigned* status;
  int n_docs;             // entries of cu - 1 (index guards of debug builds)
  int64_t n_o, n_lse;     // elements of o and lse
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint32_t tmem_base;
  int abort;
};

// Document of row t (-1 for a pad row).  Debug builds check the index into
// doc and the document's two cu_seqlens entries, and treat a row whose
// document id lies outside cu_seqlens as a pad row.
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
// One past the last row of t's document (-1 for a pad row).
__device__ __forceinline__ int64_t doc_end_of(const Params& p, int64_t t) {
  const int d = doc_index(p, t);
  if (d < 0) return -1;
  return p.cu ? (int64_t)__ldg(p.cu + d + 1) : p.S;
}

// One softmax step on this thread's S row: the 128 fp32 columns are read
// from TMEM with a single load, masked (MASK: columns outside [lo, hi] are
// -inf), reduced to the row max, and after `rescale_fn` picked the running
// max m_eff, turned into P = exp2(S*sl2 - m_eff) written as bf16 pairs over
// the first 64 columns.  Returns the fp32 row sum.
template <bool MASK, typename MaxFn>
__device__ __forceinline__ float softmax_row(uint32_t tS, int lo, int hi, float sl2,
                                             MaxFn rescale_fn) {
  uint32_t v[128];
  tc::tmem_ld_x128(tS, v);
  if (MASK) {
#pragma unroll
    for (int col = 0; col < 128; ++col)
      if (!(col >= lo && col <= hi)) v[col] = __float_as_uint(-INFINITY);
  }
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 128; i += 8) {
    m0 = tc::max3(m0, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
    m1 = tc::max3(m1, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
    m2 = tc::max3(m2, __uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]));
    m3 = tc::max3(m3, __uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
  }
  const float m_eff = rescale_fn(fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));
  float r0 = 0.f, r1 = 0.f;
#pragma unroll
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {   // pairs: one packed fma and one packed add
      float x0, x1;
      tc::fma2(x0, x1, __uint_as_float(v[c * 32 + 2 * i]), __uint_as_float(v[c * 32 + 2 * i + 1]),
               sl2, sl2, -m_eff, -m_eff);
      const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
      tc::add2(r0, r1, r0, r1, p0, p1);
      w[i] = tc::pack_bf16(p0, p1);
    }
    tc::tmem_st_x16(tS + c * 16, w);
  }
  return r0 + r1;
}

template <int D, int NH>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params p) {
  using C = Cfg<D, NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFF);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- tile coordinates (rank 0 = the last, heaviest causal query tile)
  int rank, y;
  usp::cta_coords(p.n_qtiles, p.band, rank, y);
  const int qt = p.n_qtiles - 1 - rank;
  const int per_g = p.hkv * p.slots_per_kv;
  const int g = y / per_g;
  const int jk = (y % per_g) / p.slots_per_kv;
  const int j0 = jk * p.G + (y % p.slots_per_kv) * NH;
  const int64_t t0 = (int64_t)qt * BM;

  // kv range needed by the tile: from the first row's document start up to
  // its last valid row (causal) or to the end of that row's document
  int n_kv = 0;
  int64_t kv_start = 0;
  {
    const int64_t ds0 = doc_start_of(p, t0);
    if (ds0 >= 0) {
      const int64_t last = min(t0 + BM, p.S) - 1;
      const int64_t k0 = max(ds0, p.k_lo);
      const int64_t kv_end = min(p.causal ? last + 1 : doc_end_of(p, last), p.k_hi);
      if (kv_end > k0) {
        kv_start = (k0 / BN) * BN;
        n_kv = (int)((kv_end - kv_start + BN - 1) / BN);
      }
    }
  }

  if (threadIdx.x == 0) {
    tc::mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::NSTAGE; ++s) {
      tc::mbar_init(&bars->kv_full[s], 1);
      tc::mbar_init(&bars->kv_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      tc::mbar_init(&bars->s_full[h], 1);
      tc::mbar_init(&bars->p_full[h], 128);
      tc::mbar_init(&bars->o_full[h], 1);
    }
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmV);
      tc::mbar_expect_tx(&bars->q_full, NH * C::TILE);
      for (int h = 0; h < NH; ++h)
        for (int b = 0; b < C::NB; ++b)
          tc::tma_load_3d(smem + C::Q_OFF + h * C::TILE + b * C::BOX, &tmQ, &bars->q_full,
                          (j0 + h) * D + b * 64, (int)t0, g);
      int issued = 0;
      for (int j = 0; j < n_kv && !*abort; ++j) {
        for (int w = 0; w < 2; ++w) {
          const int idx = 2 * j + w;
          const int s = idx % C::NSTAGE;
          const int use = idx / C::NSTAGE;
          if (use > 0 && !tc::mbar_wait(&bars->kv_empty[s], (use - 1) & 1, abort)) break;
          tc::mbar_expect_tx(&bars->kv_full[s], C::TILE);
          const CUtensorMap* m = w == 0 ? &tmK : &tmV;
          for (int b = 0; b < C::NB; ++b)
            tc::tma_load_3d(smem + C::KV_OFF + s * C::TILE + b * C::BOX, m, &bars->kv_full[s],
                            jk * D + b * 64, (int)(kv_start + (int64_t)j * BN), g);
          ++issued;
        }
      }
      if (*abort) {
        // let the copies already issued land before the CTA winds down
        for (int idx = (issued > C::NSTAGE ? issued - C::NSTAGE : 0); idx < issued; ++idx)
          tc::mbar_wait(&bars->kv_full[idx % C::NSTAGE], (idx / C::NSTAGE) & 1, nullptr,
                        100000000ull);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (n_kv > 0) {                    // the whole warp; one lane issues
      constexpr uint32_t idesc_qk = tc::idesc_bf16(128, BN, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(128, D, true);
      const uint32_t q_base = tc::smem_u32(smem + C::Q_OFF);
      const uint32_t kv_base = tc::smem_u32(smem + C::KV_OFF);
      // S_h = Q_h K^T for key tile `kt` (ring slot `sk`)
      auto issue_qk = [&](int h, int sk) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::BOX + (kk % 4) * 32;
          const uint64_t da = tc::desc_sw128(q_base + h * C::TILE + off, 16, 1024);
          const uint64_t db = tc::desc_sw128(kv_base + sk * C::TILE + off, 16, 1024);
          tc::mma_ss_w(tmem + C::S_COL(h), da, db, idesc_qk, kk > 0);
        }
        tc::mma_commit_w(&bars->s_full[h]);
      };
      // Issue order: QK_0(0) QK_1(0), then per key tile j
      //   PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1)
      // QK_h(j+1) rewrites S_h, which holds P_h(j): it waits for PV_h(j) to
      // complete (o_full[h]).  Each head's softmax of tile j+1 then overlaps
      // the other head's PV and QK (two MMA groups) instead of one.
      bool ok = tc::mbar_wait_warp(&bars->q_full, 0, abort) &&
                tc::mbar_wait_warp(&bars->kv_full[0], 0, abort);
      if (ok) {
        tc::fence_after_sync();
        for (int h = 0; h < NH; ++h) issue_qk(h, 0);
        tc::mma_commit_w(&bars->kv_empty[0]);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int sv = (2 * j + 1) % C::NSTAGE, uv = (2 * j + 1) / C::NSTAGE;
        const int sk = (2 * j + 2) % C::NSTAGE, uk = (2 * j + 2) / C::NSTAGE;
        const bool more = j + 1 < n_kv;
        if (!(ok = tc::mbar_wait_warp(&bars->kv_full[sv], uv & 1, abort))) break;
        for (int h = 0; h < NH && ok; ++h) {
          if (!(ok = tc::mbar_wait_warp(&bars->p_full[h], j & 1, abort))) break;
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t db = tc::desc_sw128(kv_base + sv * C::TILE + kk * 2048, C::BOX, 1024);
            tc::mma_ts_w(tmem + C::O_COL(h), tmem + C::S_COL(h) + kk * 8, db, idesc_pv,
                       (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit_w(&bars->o_full[h]);
          if (h == NH - 1) tc::mma_commit_w(&bars->kv_empty[sv]);
          if (more) {
            if (!(ok = tc::mbar_wait_warp(&bars->kv_full[sk], uk & 1, abort))) break;
            if (!(ok = tc::mbar_wait_warp(&bars->o_full[h], j & 1, abort))) break;
            tc::fence_after_sync();
            issue_qk(h, sk);
            if (h == NH - 1) tc::mma_commit_w(&bars->kv_empty[sk]);
          }
        }
      }
      if (!ok) {
        // wait (bounded) for the MMAs already issued before TMEM is freed
        tc::mma_commit_w(&bars->q_full);
        tc::mbar_wait(&bars->q_full, 1, nullptr, 100000000ull);
      }
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    const int h = (warp - 4) >> 2;        // head slot
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;    // query row within the tile
    const int64_t t = t0 + r;
    const int j = j0 + h;
    if (h < NH) {
      const int64_t ds = doc_start_of(p, t);    // -1: row sees nothing
      // visible keys [ks, ke]: from the document start (or the window start)
      // to the row itself (causal) or the document's last row, cut to the
      // key window
      const int64_t ks = max(ds, p.k_lo);
      const int64_t ke = ds < 0 ? -1 : min(p.causal ? t : doc_end_of(p, t) - 1, p.k_hi - 1);
      const uint32_t tS = tc::tmem_addr(tmem, quarter * 32, C::S_COL(h));
      const uint32_t tO = tc::tmem_addr(tmem, quarter * 32, C::O_COL(h));
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int jt = 0; jt < n_kv; ++jt) {
        ok = tc::mbar_wait_warp(&bars->s_full[h], jt & 1, abort);
        if (!ok) break;
        tc::fence_after_sync();
        const int64_t u0 = kv_start + (int64_t)jt * BN;
        const bool row_mask = ds < 0 || u0 < ks || u0 + BN - 1 > ke;
        const bool mask = __any_sync(0xffffffffu, row_mask);
        // keys u0+c visible to row t iff ks <= u0+c <= ke  (c in [lo, hi])
        const int lo = (int)max((int64_t)0, min((int64_t)BN, ks - u0));
        const int hi = ds < 0 ? -1 : (int)max((int64_t)-1, min((int64_t)BN - 1, ke - u0));
        // the mask is warp-uniform, so fully visible tiles take the path
        // without per-column tests
        bool rescale = false;
        float alpha = 1.f, m_use = m;
        auto pick = [&](float mx) {
          const float m_new = fmaxf(m, mx * p.scale_log2);
          rescale = m_new > m + kRescaleThreshold;
          m_use = rescale ? m_new : m;
          alpha = rescale ? tc::ex2(m - m_new) : 1.f;
          return m_use == -INFINITY ? 0.f : m_use;
        };
        const float rowsum = mask ? softmax_row<true>(tS, lo, hi, p.scale_log2, pick)
                                  : softmax_row<false>(tS, lo, hi, p.scale_log2, pick);
        l = l * alpha + rowsum;
        m = m_use;
        if (jt > 0 && __any_sync(0xffffffffu, rescale)) {
          ok = tc::mbar_wait_warp(&bars->o_full[h], (jt - 1) & 1, abort);
          if (!ok) break;
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tc::tmem_ld_x32(tO + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tc::tmem_st_x32(tO + c * 32, v);
          }
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        tc::mbar_arrive(&bars->p_full[h]);
      }
      // ---- epilogue: O = O / l, LSE = ln(sum)
      if (ok && n_kv > 0) {
        ok = tc::mbar_wait_warp(&bars->o_full[h], (n_kv - 1) & 1, abort);
        tc::fence_after_sync();
      }
      const bool has = ok && l > 0.f;
      const float inv = has ? 1.f / l : 0.f;
      bf16* orow = p.o + (((int64_t)g * p.S_pad + t) * p.hq + j) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        if (n_kv > 0 && ok) {
          tc::tmem_ld_x32(tO + c * 32, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = tc::pack_bf16(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
        if (t < p.S_pad && usp::in_bounds(orow + c * 32 - p.o, 32, p.n_o, p.status)) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
        }
      }
      const int64_t li = ((int64_t)g * p.hq + j) * p.S_pad + t;
      if (t < p.S_pad && usp::in_bounds(li, 1, p.n_lse, p.status))
        p.lse[li] = has ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  // ---- teardown
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  if (*abort && threadIdx.x == 0) usp::set_status(p.status, usp::kErrTimeout);
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// The driver's tensor-map encoder, looked up once per process (a
// function-local static: concurrent first calls from several host threads
// wait for one initialisation).
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

}  // namespace

// Tensor map over a head-layout tensor [P][S_pad][heads][D] (bf16) viewed as
// 3-D (heads*D, S_pad, P) with boxes of 64 columns x 128 rows, 128B swizzle.
// Rows past S_pad read as zero.
bool usp_make_head_map(CUtensorMap* map, const void* base, int heads, int D, int64_t S_pad, int P,
                       int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)heads * D, (cuuint64_t)S_pad, (cuuint64_t)P};
  cuuint64_t strides[2] = {(cuuint64_t)heads * D * 2, (cuuint64_t)S_pad * heads * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
template <int D, int NH>
cudaError_t launch_fwd(const usp::Geometry& g, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const Params& prm, cudaStream_t st) {
  using C = Cfg<D, NH>;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D, NH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int n_y = g.P * g.hkv * prm.slots_per_kv;
  const int64_t n_cta = (int64_t)prm.n_qtiles * n_y;
  if (n_cta > 0x7fffffff) return cudaErrorInvalidConfiguration;
  Params pb = prm;
  pb.band = usp::cta_band(prm.n_qtiles, n_y);
  dim3 grid((unsigned)n_cta);
  attn_fwd_tc_kernel<D, NH><<<grid, 384, C::SMEM, st>>>(mq, mk, mv, pb);
  usp_count_launches(1);
  return cudaGetLastError();
}
}  // namespace

cudaError_t usp_launch_attn_fwd(const usp::Geometry& g, const void* q, const void* k,
                                const void* v, const int32_t* doc, const int32_t* cu,
                                void* o, float* lse, cudaStream_t st, int64_t k_lo,
                                int64_t k_hi) {
  CUtensorMap mq, mk, mv;
  if (!usp_make_head_map(&mq, q, g.hq, g.D, g.S_pad, g.P, 128) ||
      !usp_make_head_map(&mk, k, g.hkv, g.D, g.S_pad, g.P, 128) ||
      !usp_make_head_map(&mv, v, g.hkv, g.D, g.S_pad, g.P, 128))
    return cudaErrorInvalidValue;
  const int nh = (g.G % 2 == 0) ? 2 : 1;
  Params prm;
  prm.doc = doc;
  prm.cu = cu;
  prm.o = reinterpret_cast<bf16*>(o);
  prm.lse = lse;
  prm.S = g.S;
  prm.S_pad = g.S_pad;
  prm.hq = g.hq;
  prm.hkv = g.hkv;
  prm.G = g.G;
  prm.n_qtiles = (int)((g.S_pad + BM - 1) / BM);
  prm.slots_per_kv = g.G / nh;
  prm.causal = g.causal;
  prm.k_lo = k_lo;
  prm.k_hi = k_hi;
  prm.scale_log2 = g.scale * kLog2e;
  prm.status = g.status;
  prm.n_docs = g.n_docs;
  prm.n_o = (int64_t)g.P * g.S_pad * g.hq * g.D;
  prm.n_lse = (int64_t)g.P * g.hq * g.S_pad;
  if (g.D == 128)
    return nh == 2 ? launch_fwd<128, 2>(g, mq, mk, mv, prm, st)
                   : launch_fwd<128, 1>(g, mq, mk, mv, prm, st);
  return nh == 2 ? launch_fwd<64, 2>(g, mq, mk, mv, prm, st)
                 : launch_fwd<64, 1>(g, mq, mk, mv, prm, st);
}
