// argus_fold_lse: fold partial attention results into an fp32 accumulator by
// their log2-sum-exp.
//
// "feat(kvcache): host-RAM KV tier for sparse-attention models", comment on
// "--kv-placement host": a deep prefill attends per 131,072-token window and
// folds the windows by their log2-sum-exp into a float32 accumulator
// (fold_attention_pass); the accumulator is allocated up front.  Per row:
//   L = max(La, Lb) + log2(2^(La - max) + 2^(Lb - max))
//   o = 2^(La - L) o_a + 2^(Lb - L) o_b,   an empty side (L = -inf) is the identity.
//
// GB300 design: an elementwise HBM stream (12 bytes per element: two reads,
// one write).  One warp owns a row so that the row's lse is read before it is
// rewritten; lanes move 16-byte float4 vectors; grid-stride over rows with the
// grid sized to the SM count.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace argus {
namespace fold {

__global__ void __launch_bounds__(256) fold_kernel(long long n_rows, int D, float* __restrict__ acc_o,
                                                   float* __restrict__ acc_lse2,
                                                   const float* __restrict__ part_o,
                                                   const float* __restrict__ part_lse2) {
  const int lane = threadIdx.x & 31;
  const long long warp = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
  const int nv = D >> 2;
  for (long long row = warp; row < n_rows; row += nwarps) {
    const float La = acc_lse2[row];
    const float Lb = __ldg(part_lse2 + row);
    if (Lb == -INFINITY) continue;  // identity
    float wa, wb, L;
    if (La == -INFINITY) {
      wa = 0.f;
      wb = 1.f;
      L = Lb;
    } else {
      const float M = fmaxf(La, Lb);
      const float ea = exp2f(La - M), eb = exp2f(Lb - M);
      L = M + log2f(ea + eb);
      wa = exp2f(La - L);
      wb = exp2f(Lb - L);
    }
    float4* a = reinterpret_cast<float4*>(acc_o + row * D);
    const float4* b = reinterpret_cast<const float4*>(part_o + row * D);
    for (int v = lane; v < nv; v += 32) {
      const float4 x = (wa == 0.f) ? make_float4(0.f, 0.f, 0.f, 0.f) : a[v];
      const float4 y = __ldg(b + v);
      a[v] = make_float4(wa * x.x + wb * y.x, wa * x.y + wb * y.y, wa * x.z + wb * y.z,
                         wa * x.w + wb * y.w);
    }
    __syncwarp();
    if (lane == 0) acc_lse2[row] = L;
  }
}

}  // namespace fold
}  // namespace argus

using namespace argus;

extern "C" argus_status argus_fold_lse(int64_t n_rows, int32_t head_dim, float* acc_o,
                                       float* acc_lse2, const float* part_o,
                                       const float* part_lse2, void* stream) {
  if (n_rows < 0 || head_dim <= 0) return fail(ARGUS_E_INVALID, "fold: negative rows or head_dim <= 0");
  if (head_dim % 4 != 0) return fail(ARGUS_E_UNSUPPORTED, "fold: head_dim %d not a multiple of 4", head_dim);
  if (n_rows == 0) return ARGUS_OK;
  if (!acc_o || !acc_lse2 || !part_o || !part_lse2) return fail(ARGUS_E_INVALID, "fold: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(acc_o) | reinterpret_cast<uintptr_t>(part_o)) & 15)
    return fail(ARGUS_E_INVALID, "fold: o arrays must be 16-byte aligned");
  const int sms = device_sm_count();
  const long long warps_needed = n_rows;
  const int blocks = (int)std::max<long long>(1, std::min<long long>((warps_needed + 7) / 8, (long long)sms * 8));
  fold::fold_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(n_rows, head_dim, acc_o, acc_lse2,
                                                                           part_o, part_lse2);
  return launch_status("argus_fold_lse");
}
