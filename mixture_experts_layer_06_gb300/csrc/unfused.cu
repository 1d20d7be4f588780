// The unfused gated activation, for the fusion ablation.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "What carries
// the argument" and the referee's minor comment 1 on the paper's section 3.3:
// the fused SwiGLU kernel is measured against running the gate and up
// projections as two GEMMs whose outputs reach global memory, then an
// element-wise SiLU(gate) * up pass.  This kernel is that pass:
// h = act(g) * u over bf16 g, u (each rounded once when the GEMMs stored
// them), computed in fp32 and rounded once to bf16.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float act_silu(float g) { return __fdividef(g, 1.f + __expf(-fmaxf(g, -80.f))); }
__device__ __forceinline__ float act_gelu(float g) { return 0.5f * g * (1.f + erff(g * 0.70710678118654752f)); }

// One thread per 8 consecutive values (16-byte loads and stores), grid-stride.
__global__ void gated_elementwise_kernel(const uint4* __restrict__ g, const uint4* __restrict__ u,
                                         uint4* __restrict__ h, size_t n8, int gelu) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 gv = g[i], uv = u[i];
    const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&gv);
    const __nv_bfloat162* up = reinterpret_cast<const __nv_bfloat162*>(&uv);
    uint4 hv;
    __nv_bfloat162* hp = reinterpret_cast<__nv_bfloat162*>(&hv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 gf = __bfloat1622float2(gp[j]), uf = __bfloat1622float2(up[j]);
      const float a0 = gelu ? act_gelu(gf.x) : act_silu(gf.x);
      const float a1 = gelu ? act_gelu(gf.y) : act_silu(gf.y);
      hp[j] = __floats2bfloat162_rn(a0 * uf.x, a1 * uf.y);
    }
    h[i] = hv;
  }
}

}  // namespace

cudaError_t launch_gated_elementwise(const void* g, const void* u, void* h, size_t n, int gelu, cudaStream_t stream) {
  const size_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  size_t blocks = (n8 + threads - 1) / threads;
  const size_t cap = static_cast<size_t>(sms) * 8;  // 8 CTAs of 256 threads per SM, grid-stride beyond
  if (blocks > cap) blocks = cap;
  return launch_kernel(gated_elementwise_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                       static_cast<const uint4*>(g), static_cast<const uint4*>(u), static_cast<uint4*>(h), n8,
                       gelu);
}

}  // namespace moe
