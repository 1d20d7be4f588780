// Weighted scatter-back of expert outputs to token order.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "The reading":
// the expert outputs are scattered back with the routing weights.  Each token
// gathers its k expert rows (through inv) instead of the rows scattering into
// the token, so no atomics are needed and the sum is taken in the fixed slot
// order j = 0..k-1 (then the shared expert) in fp32, rounded once to bf16:
// the result is bitwise deterministic.  One warp per token, 32-byte fp32
// loads and 16-byte bf16 stores.
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void combine_kernel(const float* __restrict__ y_perm, const int32_t* __restrict__ inv,
                               const float* __restrict__ topk_w, const float* __restrict__ y_shared,
                               const float* __restrict__ shared_scale, int T, int H, int k,
                               __nv_bfloat16* __restrict__ out) {
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;  // warp-uniform
  int r = -1;
  float w = 0.f;
  if (lane < k) {
    r = inv[static_cast<size_t>(t) * k + lane];
    w = topk_w[static_cast<size_t>(t) * k + lane];
  }
  const float s = shared_scale != nullptr ? shared_scale[t] : 1.f;
  for (int h0 = lane * 8; h0 < H; h0 += 256) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int rj = __shfl_sync(0xFFFFFFFFu, r, j);
      const float wj = __shfl_sync(0xFFFFFFFFu, w, j);
      if (rj < 0) continue;
      const float4* src = reinterpret_cast<const float4*>(y_perm + static_cast<size_t>(rj) * H + h0);
      const float4 a = src[0], b = src[1];
      acc[0] = fmaf(wj, a.x, acc[0]);
      acc[1] = fmaf(wj, a.y, acc[1]);
      acc[2] = fmaf(wj, a.z, acc[2]);
      acc[3] = fmaf(wj, a.w, acc[3]);
      acc[4] = fmaf(wj, b.x, acc[4]);
      acc[5] = fmaf(wj, b.y, acc[5]);
      acc[6] = fmaf(wj, b.z, acc[6]);
      acc[7] = fmaf(wj, b.w, acc[7]);
    }
    if (y_shared != nullptr) {
      const float4* src = reinterpret_cast<const float4*>(y_shared + static_cast<size_t>(t) * H + h0);
      const float4 a = src[0], b = src[1];
      acc[0] = fmaf(s, a.x, acc[0]);
      acc[1] = fmaf(s, a.y, acc[1]);
      acc[2] = fmaf(s, a.z, acc[2]);
      acc[3] = fmaf(s, a.w, acc[3]);
      acc[4] = fmaf(s, b.x, acc[4]);
      acc[5] = fmaf(s, b.y, acc[5]);
      acc[6] = fmaf(s, b.z, acc[6]);
      acc[7] = fmaf(s, b.w, acc[7]);
    }
    uint4 o;
    __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) op[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + h0) = o;
  }
}

}  // namespace

cudaError_t launch_combine(const float* y_perm, const int32_t* inv, const float* topk_w, const float* y_shared,
                           const float* shared_scale, int T, int H, int k, void* out, cudaStream_t stream) {
  const int threads = kWarpsPerBlock * 32;
  combine_kernel<<<(T + kWarpsPerBlock - 1) / kWarpsPerBlock, threads, 0, stream>>>(
      y_perm, inv, topk_w, y_shared, shared_scale, T, H, k, static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace moe
