// Weighted scatter-back of expert outputs to token order.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "The reading":
// the expert outputs are scattered back with the routing weights.  Each token
// gathers its k expert rows (through inv) instead of the rows scattering into
// the token, so no atomics are needed and the sum is taken in the fixed slot
// order j = 0..k-1 (then the shared expert) in fp32, rounded once to bf16:
// the result is bitwise deterministic.  The expert outputs arrive in fp16.
// One warp per (token, 256-column chunk), 16-byte loads and stores.
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

constexpr int kMaxSlices = 8;  // K slices of the down projection (at most 8)
constexpr long long kFewWarps = 4096;  // below this many warps the grid is latency-bound
#ifndef MOE_COMBINE_RAW
#define MOE_COMBINE_RAW 1  // many warps, one K slice: combine_raw_kernel
#endif

// 8 consecutive fp16 values (one 16-byte load) widened to fp32.
__device__ __forceinline__ void widen8(const uint4 q, float (&v)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// Sum of the nslices partial-sum slices of 8 consecutive fp16 values, in
// slice order, in fp32.  MAXS > 0: all (<= MAXS) slices are loaded before the
// first add, so their latencies overlap (for grids with few warps); MAXS ==
// 0: one slice after the other, in fewer registers (for grids with many
// warps, where occupancy hides the latency).
template <int MAXS>
__device__ __forceinline__ void load8(const __half* p, int nslices, size_t stride, float (&v)[8]) {
  if constexpr (MAXS == 0) {
    widen8(*reinterpret_cast<const uint4*>(p), v);
    for (int s = 1; s < nslices; ++s) {
      float w[8];
      widen8(*reinterpret_cast<const uint4*>(p + s * stride), w);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += w[i];
    }
  } else {
    uint4 c[MAXS];
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
      if (s < nslices) c[s] = *reinterpret_cast<const uint4*>(p + s * stride);
    widen8(c[0], v);
#pragma unroll
    for (int s = 1; s < MAXS; ++s) {
      if (s < nslices) {
        float w[8];
        widen8(c[s], w);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] += w[i];
      }
    }
  }
}

// MR / MS: load8's MAXS for the routed rows / the shared expert's row.  G:
// routed rows loaded before they are added.
template <int MR, int MS, int G>
__global__ void combine_kernel(const __half* __restrict__ y_perm, const int32_t* __restrict__ inv,
                               const float* __restrict__ topk_w, const __half* __restrict__ y_shared,
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
    // G expert rows are loaded before they are added (in slot order), so
    // their memory latencies overlap.
    for (int j0 = 0; j0 < k; j0 += G) {
      float v[G][8], wj[G];
      bool ok[G];
#pragma unroll
      for (int q = 0; q < G; ++q) {
        const int j = j0 + q;  // lanes >= k hold r = -1
        const int rj = __shfl_sync(0xFFFFFFFFu, r, j & 31);  // all lanes take part
        wj[q] = __shfl_sync(0xFFFFFFFFu, w, j & 31);
        ok[q] = j < k && rj >= 0 && active;
        if (ok[q]) load8<MR>(y_perm + static_cast<size_t>(rj) * H + h0, nslices, stride, v[q]);
      }
#pragma unroll
      for (int q = 0; q < G; ++q)
        if (ok[q]) {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[q], v[q][i], acc[i]);
        }
    }
    if (!active) return;
    if (y_shared != nullptr) {
      float v[8];
      load8<MS>(y_shared + static_cast<size_t>(t) * H + h0, nslices_sh, stride_sh, v);
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

// One K slice everywhere (large batches): all of a token's expert rows (up to
// G per round) and the shared expert's row are loaded as raw 16-byte fp16
// vectors before any of them is widened and added, so a warp keeps G + 1
// loads in flight at 4 registers each; the adds still run in slot order.
template <int G>
__global__ void combine_raw_kernel(const __half* __restrict__ y_perm, const int32_t* __restrict__ inv,
                                   const float* __restrict__ topk_w, const __half* __restrict__ y_shared,
                                   const float* __restrict__ shared_scale, int T, int H, int k,
                                   __nv_bfloat16* __restrict__ out) {
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
  const int h0 = blockIdx.y * 256 + lane * 8;  // this warp's 256-column chunk
  const bool active = h0 < H;
  uint4 sh = make_uint4(0, 0, 0, 0);
  const bool has_sh = y_shared != nullptr && active;
  if (has_sh) sh = __ldg(reinterpret_cast<const uint4*>(y_shared + static_cast<size_t>(t) * H + h0));
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < k; j0 += G) {
    uint4 raw[G];
    float wj[G];
    bool ok[G];
#pragma unroll
    for (int q = 0; q < G; ++q) {
      const int j = j0 + q;  // lanes >= k hold r = -1
      const int rj = __shfl_sync(0xFFFFFFFFu, r, j & 31);  // all lanes take part
      wj[q] = __shfl_sync(0xFFFFFFFFu, w, j & 31);
      ok[q] = j < k && rj >= 0 && active;
      if (ok[q]) raw[q] = __ldg(reinterpret_cast<const uint4*>(y_perm + static_cast<size_t>(rj) * H + h0));
    }
#pragma unroll
    for (int q = 0; q < G; ++q)
      if (ok[q]) {
        float v[8];
        widen8(raw[q], v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[q], v[i], acc[i]);
      }
  }
  if (!active) return;
  if (has_sh) {
    const float s = shared_scale != nullptr ? shared_scale[t] : 1.f;
    float v[8];
    widen8(sh, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(s, v[i], acc[i]);
  }
  uint4 o;
  __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) op[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
  *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * H + h0) = o;
}

}  // namespace

cudaError_t launch_combine(const void* y_perm, const int32_t* inv, const float* topk_w, const void* y_shared,
                           const float* shared_scale, int T, int H, int k, void* out, cudaStream_t stream,
                           int nslices, size_t slice_stride, int nslices_shared, size_t slice_stride_shared) {
  if (nslices < 1 || nslices > kMaxSlices || nslices_shared < 1 || nslices_shared > kMaxSlices)
    return cudaErrorInvalidValue;
  const int threads = kWarpsPerBlock * 32;
  const dim3 grid((T + kWarpsPerBlock - 1) / kWarpsPerBlock, (H + 255) / 256);
  // Few warps (decode-sized batches): overlap the slice loads inside each
  // warp.  Many warps with one K slice: combine_raw_kernel, every expert row
  // of a token in flight as raw fp16 (measured on GB300: DeepSeek-V3-shaped
  // T=8192 264 -> 201 us, T=2048 67 -> 53 us).  Many warps with slices: one
  // slice after the other, four expert rows in flight per warp (eight widened
  // rows measured slower: 260 -> 300 us at T=8192, at lower occupancy).
  const long long warps = static_cast<long long>(T) * grid.y;
  void (*kernel)(const __half*, const int32_t*, const float*, const __half*, const float*, int, int, int,
                 __nv_bfloat16*, int, size_t, int, size_t) = combine_kernel<0, 0, 4>;
  if (warps <= kFewWarps) {
    const bool rs = nslices > 1, ss = y_shared != nullptr && nslices_shared > 1;
    kernel = rs ? (ss ? combine_kernel<kMaxSlices, kMaxSlices, 1> : combine_kernel<kMaxSlices, 1, 1>)
                : (ss ? combine_kernel<1, kMaxSlices, 4> : combine_kernel<1, 1, 4>);
  } else if (MOE_COMBINE_RAW && nslices == 1 && (y_shared == nullptr || nslices_shared == 1)) {
    // rows in flight per round: k rounded up to 2, 4 or 8 (no unused loads or registers)
    auto raw = k <= 2 ? combine_raw_kernel<2> : k <= 4 ? combine_raw_kernel<4> : combine_raw_kernel<8>;
    return launch_kernel(raw, grid, dim3(threads), 0, stream, static_cast<const __half*>(y_perm), inv, topk_w,
                         static_cast<const __half*>(y_shared), shared_scale, T, H, k,
                         static_cast<__nv_bfloat16*>(out));
  }
  return launch_kernel(kernel, grid, dim3(threads), 0, stream, static_cast<const __half*>(y_perm), inv, topk_w,
                       static_cast<const __half*>(y_shared), shared_scale, T, H, k,
                       static_cast<__nv_bfloat16*>(out), nslices, slice_stride, nslices_shared,
                       slice_stride_shared);
}

}  // namespace moe
