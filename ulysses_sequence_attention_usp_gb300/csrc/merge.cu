// Log-sum-exp merge of partial attention results (ring attention: each ring
// step attends to one key/value chunk and yields O_i normalised within the
// chunk and LSE_i; SpecForge PR #728 and verl PR #45 configure a Ulysses x
// Ring mesh).  For every (group, row, head):
//   LSE = ln(exp(LSE_acc) + exp(LSE_i)),
//   O   = exp(LSE_acc - LSE) O_acc + exp(LSE_i - LSE) O_i,
// with the weight of a -inf term taken as 0 (both -inf: O = 0, LSE = -inf).
// The accumulator is fp32; the last step may also write O as bf16.
// HBM-bound: one group of D/4 threads per row, 16-byte fp32 / 8-byte bf16
// vectors, grid-stride.
#include "usp_common.cuh"

namespace {

using bf16 = __nv_bfloat16;

template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(
    float* __restrict__ o_acc, float* __restrict__ lse_acc, const bf16* __restrict__ o_part,
    const float* __restrict__ lse_part, int first, bf16* __restrict__ o_out, int64_t S_pad,
    int hq, int64_t n_rows, unsigned* status) {
  constexpr int TPR = D / 4;                    // threads per row
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) / TPR;
  const int sub = (int)(tid % TPR);
  for (int64_t row = tid / TPR; row < n_rows; row += stride) {
    // row = (g * S_pad + t) * hq + j ;  LSE index (g * hq + j) * S_pad + t
    const int64_t gt = row / hq;
    const int j = (int)(row - gt * hq);
    const int64_t g = gt / S_pad, t = gt - g * S_pad;
    const int64_t li = (g * hq + j) * S_pad + t;
    // index guards of debug builds: LSE arrays hold n_rows entries, O arrays n_rows*D
    if (!usp::in_bounds(li, 1, n_rows, status) ||
        !usp::in_bounds(row * D + 4 * sub, 4, n_rows * D, status))
      continue;
    const float lb = __ldg(lse_part + li);
    const float la = first ? -INFINITY : lse_acc[li];
    const float mx = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f, l = -INFINITY;
    if (mx != -INFINITY) {
      const float ea = expf(la - mx), eb = expf(lb - mx);   // exp(-inf) = 0
      const float z = ea + eb;
      l = mx + logf(z);
      wa = ea / z;
      wb = eb / z;
    }
    const uint2 pb = __ldg(reinterpret_cast<const uint2*>(o_part + row * D) + sub);
    const float2 b01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pb.x));
    const float2 b23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pb.y));
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!first) a = reinterpret_cast<const float4*>(o_acc + row * D)[sub];
    float4 r;
    r.x = wb == 0.f ? wa * a.x : fmaf(wb, b01.x, wa * a.x);
    r.y = wb == 0.f ? wa * a.y : fmaf(wb, b01.y, wa * a.y);
    r.z = wb == 0.f ? wa * a.z : fmaf(wb, b23.x, wa * a.z);
    r.w = wb == 0.f ? wa * a.w : fmaf(wb, b23.y, wa * a.w);
    reinterpret_cast<float4*>(o_acc + row * D)[sub] = r;
    if (sub == 0) lse_acc[li] = l;
    if (o_out != nullptr) {
      const __nv_bfloat162 c01 = __floats2bfloat162_rn(r.x, r.y);
      const __nv_bfloat162 c23 = __floats2bfloat162_rn(r.z, r.w);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&c01);
      w.y = *reinterpret_cast<const uint32_t*>(&c23);
      reinterpret_cast<uint2*>(o_out + row * D)[sub] = w;
    }
  }
}

}  // namespace

cudaError_t usp_launch_lse_merge(const usp::Geometry& g, float* o_acc, float* lse_acc,
                                 const void* o_part, const float* lse_part, int first,
                                 void* o_out, cudaStream_t st) {
  const int64_t n_rows = (int64_t)g.P * g.S_pad * g.hq;
  const int64_t threads = n_rows * (g.D / 4);
  int64_t blocks = (threads + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  const bf16* pb = reinterpret_cast<const bf16*>(o_part);
  bf16* ob = reinterpret_cast<bf16*>(o_out);
  if (g.D == 128)
    lse_merge_kernel<128><<<(int)blocks, 256, 0, st>>>(o_acc, lse_acc, pb, lse_part, first, ob,
                                                       g.S_pad, g.hq, n_rows, g.status);
  else
    lse_merge_kernel<64><<<(int)blocks, 256, 0, st>>>(o_acc, lse_acc, pb, lse_part, first, ob,
                                                      g.S_pad, g.hq, n_rows, g.status);
  usp_count_launches(1);
  return cudaGetLastError();
}
