// Router scoring + top-k selection.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "The reading":
// every token is first scored by the router.  Here the scoring GEMM
// logits[T, E] = x[T, H] . W_r[E, H]^T runs on the 5th-generation tensor
// cores (tcgen05.mma, operands staged by TMA, fp32 accumulator in TMEM), and
// the epilogue reads each token's E logits straight out of its TMEM lane:
// one thread per token applies the logit bias, the score function (softmax or
// sigmoid), optional group limiting, and keeps the k best experts in
// registers.  Nothing but topk_idx / topk_w is written to global memory.
#include <cfloat>

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;  // warp 0: TMA, warp 1: MMA + TMEM owner, warps 2-5: epilogue
constexpr int kMaxStages = 8;
constexpr int kTileM = 128;    // tokens per CTA
constexpr int kTileK = 64;     // bf16 elements per 128-byte swizzled row
constexpr int kATileBytes = kTileM * kTileK * 2;

struct RouterArgs {
  int T, H, E, k, NE, stages, tmem_cols;
  RouteSpec spec;
  int32_t* topk_idx;
  float* topk_w;
  uint32_t* err;
};

// Keep the KMAX largest values seen so far, sorted descending; a value equal
// to one already kept goes after it (so earlier = lower index wins ties).
template <int KMAX>
__device__ __forceinline__ void keep_top(float (&bv)[KMAX], int (&bi)[KMAX], float v, int e) {
#pragma unroll
  for (int j = KMAX - 1; j >= 0; --j) {
    if (v > bv[j]) {
      if (j > 0 && v > bv[j - 1]) {
        bv[j] = bv[j - 1];
        bi[j] = bi[j - 1];
      } else {
        bv[j] = v;
        bi[j] = e;
      }
    }
  }
}

// Load TMEM columns [c0, c0+32) (or 16 when only 16 remain) of this warp's lanes.
__device__ __forceinline__ void load_chunk(uint32_t taddr, int remaining, uint32_t (&r)[32]) {
  if (remaining >= 32)
    tmem_ld32(taddr, r);
  else
    tmem_ld16(taddr, r);
  tmem_wait(r);
}

template <int KMAX>
__device__ void router_epilogue(const RouterArgs& a, uint32_t tmem_base, const float* bias_s, int m0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  const int row = m0 + q * 32 + lane;
  const uint32_t tbase = tmem_addr(tmem_base, q * 32, 0);
  const int E = a.E, NE = a.NE;
  const bool sigmoid = a.spec.sigmoid != 0;

  // Pass 1: max and sum of exp over all E logits (softmax normaliser).
  float mx = -FLT_MAX, se = 0.f;
  for (int c0 = 0; c0 < NE; c0 += 32) {
    uint32_t r[32];
    load_chunk(tbase + c0, NE - c0, r);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = c0 + i;
      if (e < E) {
        const float l = __uint_as_float(r[i]) + bias_s[e];
        if (l > mx) {
          se = se * __expf(mx - l) + 1.f;
          mx = l;
        } else {
          se += __expf(l - mx);
        }
      }
    }
  }
  const float inv_se = 1.f / se;

  // Pass 2 (group-limited routing): group scores and the kept-group mask.
  uint32_t kept = 0xFFFFFFFFu;
  int gsize = E;
  if (a.spec.n_group > 1) {
    gsize = E / a.spec.n_group;
    float gsc[16];
    float top[4] = {-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX};
    int topi[4] = {0, 0, 0, 0};
    int g = 0, gi = 0;
    for (int c0 = 0; c0 < NE; c0 += 32) {
      uint32_t r[32];
      load_chunk(tbase + c0, NE - c0, r);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = c0 + i;
        if (e < E) {
          const float l = __uint_as_float(r[i]) + bias_s[e];
          const float sc = sigmoid ? 1.f / (1.f + __expf(-l)) : __expf(l - mx) * inv_se;
          keep_top<4>(top, topi, sc, e);
          if (++gi == gsize) {
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j < a.spec.group_topn) sum += top[j];
            gsc[g++] = sum;
            gi = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) top[j] = -FLT_MAX;
          }
        }
      }
    }
    kept = 0;
    for (int rsel = 0; rsel < a.spec.topk_group; ++rsel) {
      int best = -1;
      float bestv = -FLT_MAX;
      for (int gg = 0; gg < a.spec.n_group; ++gg) {
        if ((kept >> gg) & 1u) continue;
        if (best < 0 || gsc[gg] > bestv) {
          best = gg;
          bestv = gsc[gg];
        }
      }
      kept |= 1u << best;
    }
  }

  // Pass 3: the KMAX best candidate logits (score functions are monotone).
  float bv[KMAX];
  int bi[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    bv[j] = -FLT_MAX;
    bi[j] = 0;
  }
  {
    int g = 0, gi = 0;
    for (int c0 = 0; c0 < NE; c0 += 32) {
      uint32_t r[32];
      load_chunk(tbase + c0, NE - c0, r);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = c0 + i;
        if (e < E) {
          if ((kept >> g) & 1u) keep_top<KMAX>(bv, bi, __uint_as_float(r[i]) + bias_s[e], e);
          if (++gi == gsize) {
            gi = 0;
            ++g;
          }
        }
      }
    }
  }

  if (row < a.T) {
    float sc[KMAX];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      sc[j] = sigmoid ? 1.f / (1.f + __expf(-bv[j])) : __expf(bv[j] - mx) * inv_se;
      if (j < a.k) sum += sc[j];
    }
    const float scale = a.spec.renormalize ? a.spec.route_scale / sum : a.spec.route_scale;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < a.k) {
        a.topk_idx[static_cast<size_t>(row) * a.k + j] = bi[j];
        a.topk_w[static_cast<size_t>(row) * a.k + j] = sc[j] * scale;
      }
    }
  }
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1)
    router_topk_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_wr,
                       const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const int b_tile_bytes = a.NE * kTileK * 2;
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kATileBytes;
  float* bias_s = reinterpret_cast<float*>(sB + S * b_tile_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(bias_s + 256);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kTileM;
  const int KB = a.H / kTileK;

  for (int e = threadIdx.x; e < 256; e += kThreads)
    bias_s[e] = (a.spec.logit_bias != nullptr && e < a.E) ? a.spec.logit_bias[e] : 0.f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
    tma_prefetch_map(&map_x);
    tma_prefetch_map(&map_wr);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t bytes = kATileBytes + b_tile_bytes;
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % S;
        const uint32_t ph = (kb / S) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, a.err, kSiteRouterProducer)) break;
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_2d(sA + s * kATileBytes, &map_x, &full[s], kb * kTileK, m0);
        tma_load_2d(sB + s * b_tile_bytes, &map_wr, &full[s], kb * kTileK, 0);
        ++issued;
      }
      // Do not leave while copies into this CTA's shared memory are in flight.
      for (int kb = (issued > S ? issued - S : 0); kb < issued; ++kb)
        mbar_wait(&full[kb % S], (kb / S) & 1, a.err, kSiteTeardown);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, a.NE);
      bool ok = true;
      for (int kb = 0; kb < KB && ok; ++kb) {
        const int s = kb % S;
        const uint32_t ph = (kb / S) & 1;
        if (!mbar_wait(&full[s], ph, a.err, kSiteRouterMma)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(sA + s * kATileBytes);
        const uint32_t b_addr = smem_u32(sB + s * b_tile_bytes);
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk)
          umma_bf16(tmem_base, sdesc_k128(a_addr + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                    (kb | kk) != 0);
        umma_commit(&empty[s]);
      }
      umma_commit(acc_full);
    }
  } else {
    if (mbar_wait(acc_full, 0, a.err, kSiteRouterEpilogue)) {
      tc_fence_after_sync();
      router_epilogue<KMAX>(a, tmem_base, bias_s, m0);
    }
    tc_fence_before_sync();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

// shared_scale[t] = sigmoid(x[t] . w_s): one warp per token, 16-byte loads.
__global__ void shared_gate_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ ws, int T,
                                   int H, float* __restrict__ scale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= T) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(warp) * H);
  const uint4* wr = reinterpret_cast<const uint4*>(ws);
  float acc = 0.f;
  for (int v = lane; v < H / 8; v += 32) {
    const uint4 xa = xr[v], wa = wr[v];
    const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xa);
    const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wa);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 xf = __bfloat1622float2(xp[i]), wf = __bfloat1622float2(wp[i]);
      acc = fmaf(xf.x, wf.x, acc);
      acc = fmaf(xf.y, wf.y, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) scale[warp] = 1.f / (1.f + __expf(-acc));
}

template <int KMAX>
cudaError_t launch_router_k(const CUtensorMap& mx, const CUtensorMap& mw, const RouterArgs& a, size_t smem,
                            cudaStream_t stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_topk_kernel<KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int grid = (a.T + kTileM - 1) / kTileM;
  router_topk_kernel<KMAX><<<grid, kThreads, smem, stream>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_wr, int T, int H, int E, int k,
                          const RouteSpec& spec, int32_t* topk_idx, float* topk_w, uint32_t* err,
                          cudaStream_t stream) {
  RouterArgs a{};
  a.T = T;
  a.H = H;
  a.E = E;
  a.k = k;
  a.NE = (E + 15) / 16 * 16;
  a.tmem_cols = a.NE <= 32 ? 32 : a.NE <= 64 ? 64 : a.NE <= 128 ? 128 : 256;
  a.spec = spec;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.err = err;
  const int stage_bytes = kATileBytes + a.NE * kTileK * 2;
  const int fixed = 1024 + 256 * 4 + (2 * kMaxStages + 2) * 8 + 64;
  int stages = (227 * 1024 - fixed) / stage_bytes;
  const int KB = H / kTileK;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages > KB) stages = KB;
  a.stages = stages;
  const size_t smem = static_cast<size_t>(fixed) + static_cast<size_t>(stages) * stage_bytes;
  if (k <= 2) return launch_router_k<2>(map_x, map_wr, a, smem, stream);
  if (k <= 4) return launch_router_k<4>(map_x, map_wr, a, smem, stream);
  if (k <= 8) return launch_router_k<8>(map_x, map_wr, a, smem, stream);
  return launch_router_k<16>(map_x, map_wr, a, smem, stream);
}

cudaError_t launch_shared_gate(const void* x, const void* w_s, int T, int H, float* shared_scale,
                               cudaStream_t stream) {
  const int threads = 256;
  const int grid = (T * 32 + threads - 1) / threads;
  shared_gate_kernel<<<grid, threads, 0, stream>>>(static_cast<const __nv_bfloat16*>(x),
                                                   static_cast<const __nv_bfloat16*>(w_s), T, H, shared_scale);
  return cudaGetLastError();
}

}  // namespace moe
