// Router scoring + top-k selection.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "The reading":
// every token is first scored by the router; "Assumptions & free parameters":
// the standard softmax/sigmoid router with top-k selection.
//
// Two launches:
//  1. router_gemm_kernel: logits = x . [W_r; w_s]^T on the 5th-generation
//     tensor cores (tcgen05.mma, operands staged by TMA, fp32 accumulator in
//     TMEM).  The grid is (token tiles of 128) x (K slices), so that even a
//     single token spreads the W_r stream over many SMs; each CTA writes its
//     fp32 partial logits to a slice of the scratch.  With a sigmoid-gated
//     shared expert the gate vector w_s rides along as one more B row.
//  2. router_topk_kernel: one warp per token adds the K-slice partials in
//     slice order, applies the logit bias and the score function, optional
//     group limiting, and picks the k best experts by warp-wide arg-max
//     rounds (ties to the lower expert index).  Deterministic.
#include <cfloat>
#include <climits>

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 192;  // warp 0: TMA, warp 1: MMA + TMEM owner, warps 2-5: epilogue
constexpr int kMaxStages = 8;
constexpr int kTileM = 128;    // tokens per CTA
constexpr int kTileK = 64;     // bf16 elements per 128-byte swizzled row
constexpr int kATileBytes = kTileM * kTileK * 2;
constexpr int kBoxBytes = 16 * kTileK * 2;  // one 16-row box of B rows
constexpr int kJMax = 8;                    // logit columns per lane in the top-k kernel (<= 256 columns)

struct GemmArgs {
  int T, H, NE, n_wr_boxes, gate_box, stages, tmem_cols, kb_per_split;
  float* partial;  // [ksplit][T][NE]
  uint32_t* err;
};

__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_wr,
                       const __grid_constant__ CUtensorMap map_ws, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const int stage_bytes = kATileBytes + a.NE * kTileK * 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * stage_bytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kTileM;
  const int ks = blockIdx.y;
  const int KB = a.H / kTileK;
  const int kb0 = ks * a.kb_per_split;
  const int kb1 = min(KB, kb0 + a.kb_per_split);
  const int nboxes = a.n_wr_boxes + (a.gate_box >= 0 ? 1 : 0);

  pdl_trigger();
  // x and the partial-logit scratch belong to earlier work of the stream;
  // waiting before the TMEM allocation also means a kernel never holds TMEM
  // while an earlier one on the same SM may still need some.
  pdl_wait();
  if (threadIdx.x == 64) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
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
    // Lane 0: wait for the slot, post the bytes, load the x tile, the W_r rows
    // (one box) and, with a fused gate, the w_s row (one 16-row box).
    if (lane == 0) {
      int issued = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++issued) {
        const int s = issued % S;
        const uint32_t ph = (issued / S) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, a.err, kSiteRouterProducer)) break;
        mbar_arrive_expect_tx(&full[s], kATileBytes + nboxes * kBoxBytes);
        uint8_t* st = smem + s * stage_bytes;
        tma_load_2d(st, &map_x, &full[s], kb * kTileK, m0);
        tma_load_2d(st + kATileBytes, &map_wr, &full[s], kb * kTileK, 0);
        if (a.gate_box >= 0) tma_load_2d(st + kATileBytes + a.gate_box * kBoxBytes, &map_ws, &full[s], kb * kTileK, 0);
      }
      // Do not leave while copies into this CTA's shared memory are in flight.
      for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
        mbar_wait(&full[i % S], (i / S) & 1, a.err, kSiteTeardown);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, a.NE);
      int n = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++n) {
        const int s = n % S;
        if (!mbar_wait(&full[s], (n / S) & 1, a.err, kSiteRouterMma)) break;
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(smem + s * stage_bytes);
        const uint32_t b_addr = a_addr + kATileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk)
          umma_bf16(tmem_base, sdesc_k128(a_addr + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                    (kb != kb0 || kk != 0));
        umma_commit(&empty[s]);
      }
      umma_commit(acc_full);
    }
  } else {
    // Epilogue: thread = token row (TMEM lane); write its NE partial logits.
    if (mbar_wait(acc_full, 0, a.err, kSiteRouterEpilogue)) {
      tc_fence_after_sync();
      const int q = warp & 3;
      const int row = m0 + q * 32 + lane;
      float* dst = a.partial + (static_cast<size_t>(ks) * a.T + row) * a.NE;
      for (int c0 = 0; c0 < a.NE; c0 += 32) {
        uint32_t r[32];
        const uint32_t ta = tmem_addr(tmem_base, q * 32, c0);
        if (a.NE - c0 >= 32)
          tmem_ld32(ta, r);
        else
          tmem_ld16(ta, r);
        tmem_wait(r);
        const int nc = min(32, a.NE - c0);
        if (row < a.T) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            if (i < nc)
              *reinterpret_cast<float4*>(dst + c0 + i) = make_float4(
                  __uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
        }
      }
    }
    tc_fence_before_sync();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

// Warp-wide arg-max: the larger value wins, equal values go to the lower index.
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (v2 > v || (v2 == v && i2 < i)) {
      v = v2;
      i = i2;
    }
  }
}

struct TopkArgs {
  const float* partial;
  int ksplit, T, NE, E, k, gate_col;
  RouteSpec spec;
  int32_t* topk_idx;
  float* topk_w;
  float* shared_scale;
};

__global__ void router_topk_kernel(const TopkArgs a) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= a.T) return;  // warp-uniform
  const int E = a.E;
  const bool sigmoid = a.spec.sigmoid != 0;

  // Logit column c = lane + 32 j lives in l[j]; partials added in slice order.
  float l[kJMax];
#pragma unroll
  for (int j = 0; j < kJMax; ++j) {
    const int c = lane + 32 * j;
    float v = -INFINITY;
    if (c < a.NE) {
      v = 0.f;
      for (int s = 0; s < a.ksplit; ++s) v += a.partial[(static_cast<size_t>(s) * a.T + t) * a.NE + c];
      if (c == a.gate_col) a.shared_scale[t] = 1.f / (1.f + __expf(-v));
      if (c < E) {
        if (a.spec.logit_bias != nullptr) v += a.spec.logit_bias[c];
      } else {
        v = -INFINITY;
      }
    }
    l[j] = v;
  }

  // Softmax normaliser over all E logits (fixed butterfly order).
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < kJMax; ++j) mx = fmaxf(mx, l[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  float se = 0.f;
#pragma unroll
  for (int j = 0; j < kJMax; ++j)
    if (lane + 32 * j < E) se += __expf(l[j] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xFFFFFFFFu, se, o);
  const float inv_se = 1.f / se;
  auto score = [&](float v) { return sigmoid ? 1.f / (1.f + __expf(-v)) : __expf(v - mx) * inv_se; };

  // Group limiting: group score = sum of its top group_topn scores; keep the
  // topk_group best groups (lane g holds group g's score).  Scores and group
  // ids are computed once per column.
  const int gsize = a.spec.n_group > 1 ? E / a.spec.n_group : E;
  uint32_t kept = 0xFFFFFFFFu;
  int gid[kJMax];
  if (a.spec.n_group > 1) {
    float sc[kJMax];
#pragma unroll
    for (int j = 0; j < kJMax; ++j) {
      const int c = lane + 32 * j;
      sc[j] = c < E ? score(l[j]) : -INFINITY;
      gid[j] = c < E ? c / gsize : -1;  // no group
    }
    float my_gscore = -INFINITY;
    if (gsize % 32 == 0 && a.spec.group_topn <= 2) {
      // Group g is the columns j in [g*gpj, (g+1)*gpj) of every lane: each
      // lane takes its own best two, then a butterfly merges the pairs
      // (disjoint lane sets at every step, so nothing is counted twice).
      const int gpj = gsize / 32;
      for (int g = 0; g < a.spec.n_group; ++g) {
        float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
        for (int j = 0; j < kJMax; ++j) {
          if (j >= g * gpj && j < (g + 1) * gpj) {
            const float v = sc[j];
            if (v > b1) {
              b2 = b1;
              b1 = v;
            } else if (v > b2) {
              b2 = v;
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float p1 = __shfl_xor_sync(0xFFFFFFFFu, b1, o), p2 = __shfl_xor_sync(0xFFFFFFFFu, b2, o);
          if (b1 >= p1) {
            b2 = fmaxf(b2, p1);
          } else {
            b2 = fmaxf(p2, b1);
            b1 = p1;
          }
        }
        const float sum = a.spec.group_topn == 2 ? b1 + b2 : b1;
        if (lane == g) my_gscore = sum;
      }
    } else {
      for (int g = 0; g < a.spec.n_group; ++g) {
        uint32_t taken = 0;
        float sum = 0.f;
        for (int r = 0; r < a.spec.group_topn; ++r) {
          float v = -INFINITY;
          int i = INT_MAX;
#pragma unroll
          for (int j = 0; j < kJMax; ++j) {
            const int c = lane + 32 * j;
            if (gid[j] == g && !((taken >> j) & 1u) && (sc[j] > v || (sc[j] == v && c < i))) {
              v = sc[j];
              i = c;
            }
          }
          warp_best(v, i);
          sum += v;
          if (i != INT_MAX && (i & 31) == lane) taken |= 1u << (i >> 5);
        }
        if (lane == g) my_gscore = sum;
      }
    }
    kept = 0;
    for (int r = 0; r < a.spec.topk_group; ++r) {
      float v = (lane < a.spec.n_group && !((kept >> lane) & 1u)) ? my_gscore : -INFINITY;
      int i = lane < a.spec.n_group ? lane : INT_MAX;
      warp_best(v, i);
      if (i != INT_MAX) kept |= 1u << i;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kJMax; ++j) gid[j] = 0;
  }

  // k rounds of warp arg-max over the candidate logits (the score functions
  // are monotone, so ordering by logit is ordering by score).
  uint32_t taken = 0;
  int my_idx = 0;
  float my_score = 0.f, sum = 0.f;
  for (int r = 0; r < a.k; ++r) {
    float v = -INFINITY;
    int i = INT_MAX;
#pragma unroll
    for (int j = 0; j < kJMax; ++j) {
      const int c = lane + 32 * j;
      if (c < E && ((kept >> gid[j]) & 1u) && !((taken >> j) & 1u)) {
        if (l[j] > v || (l[j] == v && c < i)) {
          v = l[j];
          i = c;
        }
      }
    }
    warp_best(v, i);
    if (i != INT_MAX && (i & 31) == lane) taken |= 1u << (i >> 5);
    const float sc = score(v);
    sum += sc;
    if (lane == r) {
      my_idx = i;
      my_score = sc;
    }
  }
  if (lane < a.k) {
    const float scale = a.spec.renormalize ? a.spec.route_scale / sum : a.spec.route_scale;
    a.topk_idx[static_cast<size_t>(t) * a.k + lane] = my_idx;
    a.topk_w[static_cast<size_t>(t) * a.k + lane] = my_score * scale;
  }
}

// shared_scale[t] = sigmoid(x[t] . w_s): one warp per token, 16-byte loads.
// Used only when the gate vector does not fit as an extra router B row.
__global__ void shared_gate_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ ws, int T,
                                   int H, float* __restrict__ scale) {
  pdl_trigger();
  pdl_wait();
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

}  // namespace

RouterPlan router_plan(int T, int H, int E, bool shared_gate) {
  RouterPlan p{};
  const int ne_wr = (E + 15) / 16 * 16;
  p.fused_gate = shared_gate && ne_wr + 16 <= 256;
  p.NE = ne_wr + (p.fused_gate ? 16 : 0);
  const int m_tiles = (T + kTileM - 1) / kTileM;
  const int KB = H / kTileK;
  // Enough K slices to put ~152 CTAs to work, at least 2 k-blocks each, and at
  // most ~32 MB of partial logits.  Depends on the shapes only.
  int ks = 152 / (m_tiles > 0 ? m_tiles : 1);
  if (ks > KB / 2) ks = KB / 2;
  const long long per_slice = static_cast<long long>(T) * p.NE * 4;
  if (per_slice > 0 && ks * per_slice > (32ll << 20)) ks = static_cast<int>((32ll << 20) / per_slice);
  if (ks < 1) ks = 1;
  const int kbs = (KB + ks - 1) / ks;
  p.ksplit = (KB + kbs - 1) / kbs;
  p.kb_per_split = kbs;
  p.scratch_bytes = static_cast<size_t>(p.ksplit) * per_slice;
  return p;
}

cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_wr, const CUtensorMap* map_ws, int T,
                          int H, int E, int k, const RouteSpec& spec, const void* x, const void* w_shared_gate,
                          int32_t* topk_idx, float* topk_w, float* shared_scale, void* scratch, uint32_t* err,
                          cudaStream_t stream) {
  const RouterPlan p = router_plan(T, H, E, w_shared_gate != nullptr && shared_scale != nullptr);
  GemmArgs g{};
  g.T = T;
  g.H = H;
  g.NE = p.NE;
  g.n_wr_boxes = (E + 15) / 16;
  g.gate_box = p.fused_gate ? g.n_wr_boxes : -1;
  g.tmem_cols = p.NE <= 32 ? 32 : p.NE <= 64 ? 64 : p.NE <= 128 ? 128 : 256;
  g.kb_per_split = p.kb_per_split;
  g.partial = static_cast<float*>(scratch);
  g.err = err;
  const int stage_bytes = kATileBytes + p.NE * kTileK * 2;
  const int fixed = 1024 + (2 * kMaxStages + 2) * 8 + 64;
  int stages = (227 * 1024 - fixed) / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages > p.kb_per_split) stages = p.kb_per_split;
  g.stages = stages;
  const size_t smem = static_cast<size_t>(fixed) + static_cast<size_t>(stages) * stage_bytes;

  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const dim3 grid((T + kTileM - 1) / kTileM, p.ksplit);
  cudaError_t e = launch_kernel(router_gemm_kernel, grid, dim3(kThreads), smem, stream, map_x, map_wr,
                                p.fused_gate ? *map_ws : map_wr, g);
  if (e != cudaSuccess) return e;

  TopkArgs t{};
  t.partial = g.partial;
  t.ksplit = p.ksplit;
  t.T = T;
  t.NE = p.NE;
  t.E = E;
  t.k = k;
  t.gate_col = p.fused_gate ? g.n_wr_boxes * 16 : -1;
  t.spec = spec;
  t.topk_idx = topk_idx;
  t.topk_w = topk_w;
  t.shared_scale = shared_scale;
  const int warps = 8;
  e = launch_kernel(router_topk_kernel, dim3((T + warps - 1) / warps), dim3(warps * 32), 0, stream, t);
  if (e != cudaSuccess) return e;
  if (w_shared_gate != nullptr && shared_scale != nullptr && !p.fused_gate) {
    e = launch_kernel(shared_gate_kernel, dim3((T * 32 + 255) / 256), dim3(256), 0, stream,
                      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_shared_gate), T, H,
                      shared_scale);
  }
  return e;
}

}  // namespace moe
