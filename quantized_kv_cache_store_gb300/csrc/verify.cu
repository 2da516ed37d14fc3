// verify.cu -- spec-verify stage 2: the log-sum-exp merge of the split-KV
// partials ("sycl-three-attempts-arc-b70", section "Part 3: joint_matrix +
// split-KV"; "spec-decode-intel-arc", section "Roofline": the stage-2
// reduction kernel), and the stage-1 dispatch to the tensor-core kernel.
//   out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M),  M = max_s lse_s,
// and out = 0 for a row whose splits are all empty.
#include <math_constants.h>

#include "tq_common.cuh"

namespace tq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---- stage 2: one warp per (n, b, h) row, lane owns 4 coordinates; lane s
// owns split s's weight exp(lse_s - M), broadcast while the partial rows of
// eight splits are loaded back to back
__global__ void __launch_bounds__(128) verify_stage2_kernel(MergeArgs a) {
  pdl_wait();
  pdl_trigger();
  const long row = (long)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  const float* lse = a.part_lse + row * a.S;
  float M = -CUDART_INF_F;
  for (int s = lane; s < a.S; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -CUDART_INF_F) {
    const float* po = a.part_o + row * a.S * kD + 4 * lane;
    float den = 0.f;
    for (int s0 = 0; s0 < a.S; s0 += 32) {
      const int s = s0 + lane;
      const float l = s < a.S ? lse[s] : -CUDART_INF_F;
      const float wl = l == -CUDART_INF_F ? 0.f : expf(l - M);
      den += wl;
      const int n = min(32, a.S - s0);
#pragma unroll 8
      for (int k = 0; k < n; ++k) {
        const float w = __shfl_sync(kFull, wl, k);
        const float4 v = *reinterpret_cast<const float4*>(po + (long)(s0 + k) * kD);
        if (w != 0.f) {  // an empty split contributes nothing
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
          acc.z = fmaf(w, v.z, acc.z);
          acc.w = fmaf(w, v.w, acc.w);
        }
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
    const float inv = 1.f / den;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
  }
  *reinterpret_cast<float4*>(a.out + row * kD + 4 * lane) = acc;
}

}  // namespace

cudaError_t launch_verify_stage1(int preset, const VerifyArgs& a, cudaStream_t st) {
  return launch_verify_stage1_tc(preset, a, st);
}

cudaError_t launch_verify_stage2(const MergeArgs& a, cudaStream_t st) {
  if (a.rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((a.rows + 3) / 4);
  return launch_pdl(verify_stage2_kernel, dim3(grid), dim3(128), 0, st, a);
}

}  // namespace tq
