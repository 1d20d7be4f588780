// Weighted scatter-back of expert outputs to token order.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "The reading":
// the expert outputs are scattered back with the routing weights.  Each token
// gathers its k expert rows (through inv) instead of the rows scattering into
// the token, so no atomics are needed and the sum is taken in the fixed slot
// order j = 0..k-1 (then the shared expert) in fp32, rounded once to bf16:
// the result is bitwise deterministic.  One warp per (token, 256-column
// chunk), 32-byte fp32 loads and 16-byte bf16 stores.
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

// Sum of the nslices partial-sum slices of 8 consecutive fp32 values, in
// slice order.
__device__ __forceinline__ void load8(const float* p, int nslices, size_t stride, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  for (int s = 1; s < nslices; ++s) {
    const float4* q = reinterpret_cast<const float4*>(p + s * stride);
    const float4 c = q[0], d = q[1];
    v[0] += c.x; v[1] += c.y; v[2] += c.z; v[3] += c.w;
    v[4] += d.x; v[5] += d.y; v[6] += d.z; v[7] += d.w;
  }
}

__global__ void combine_kernel(const float* __restrict__ y_perm, const int32_t* __restrict__ inv,
                               const float* __restrict__ topk_w, const float* __restrict__ y_shared,
                               const float* __restrict__ shared_scale, int T, int H, int k,
                               __nv_bfloat16* __restrict__ out, int nslices, size_t stride, int nslices_sh,
                               size_t stride_sh) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;  // warp-uniform
  int r = -1;
  float w = 0.f;
  if (lane < k) {
    r = inv[static_cast<size_t>(t) * k + lane];
    w = topk_w[static_cast<size_t>(t) * k + lane];
  }
  const float s = shared_scale != nullptr ? shared_scale[t] : 1.f;
  const int h0 = blockIdx.y * 256 + lane * 8;  // this warp's 256-column chunk
  const bool active = h0 < H;
  {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int rj = __shfl_sync(0xFFFFFFFFu, r, j);  // all lanes take part
      const float wj = __shfl_sync(0xFFFFFFFFu, w, j);
      if (rj < 0 || !active) continue;
      float v[8];
      load8(y_perm + static_cast<size_t>(rj) * H + h0, nslices, stride, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[i], acc[i]);
    }
    if (!active) return;
    if (y_shared != nullptr) {
      float v[8];
      load8(y_shared + static_cast<size_t>(t) * H + h0, nslices_sh, stride_sh, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(s, v[i], acc[i]);
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
                           const float* shared_scale, int T, int H, int k, void* out, cudaStream_t stream,
                           int nslices, size_t slice_stride, int nslices_shared, size_t slice_stride_shared) {
  const int threads = kWarpsPerBlock * 32;
  const dim3 grid((T + kWarpsPerBlock - 1) / kWarpsPerBlock, (H + 255) / 256);
  return launch_kernel(combine_kernel, grid, dim3(threads), 0, stream, y_perm, inv, topk_w, y_shared, shared_scale, T,
                       H, k, static_cast<__nv_bfloat16*>(out), nslices, slice_stride, nslices_shared,
                       slice_stride_shared);
}

}  // namespace moe
