// Host-side launchers of the MoE kernels (internal to the library).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

// Kernel launch on `stream` with programmatic dependent launch (the kernel
// starts launching while the previous kernel of the stream finishes and
// waits for it with pdl_wait before touching global memory).  MOE_PDL=0 at
// build time launches with plain stream order.
#ifndef MOE_PDL
#define MOE_PDL 1
#endif
// Kernels launched through launch_kernel since the library was loaded.
extern std::atomic<unsigned long long> g_launch_count;

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// launch_kernel for a grid of thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                  unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// Routing variant as the kernels see it.
struct RouteSpec {
  int sigmoid;       // 0 softmax, 1 sigmoid
  int renormalize;
  float route_scale;
  int n_group;       // <= 1: off
  int topk_group;
  int group_topn;
  const float* logit_bias;  // [E] or nullptr
};

// Router launch plan: logit columns NE (E rounded up to 16, plus 16 when the
// shared-expert gate vector rides along as one more B row), and the K split:
// ksplit CTAs (or CTA pairs, `pair`) per token tile of 128 (256) tokens, each
// reducing kb_per_cta 64-wide K blocks; a cluster of `cluster` CTAs per tile.
// With pairs, map_wr's box is NE/2 rows.  Shapes only.
struct RouterPlan {
  bool fused_gate;
  bool pair;
  int NE;
  int ksplit;
  int cluster;
  int kb_per_cta;
  int m_tiles;
};
RouterPlan router_plan(int T, int H, int E, bool shared_gate);

// Router scoring + top-k in one launch (x [T,H] . [W_r; w_s]^T on the tensor
// cores, partial logits of the cluster added over distributed shared memory,
// then score, group limit and top-k per token), plus the separate shared-gate
// kernel when the gate row does not fit.  map_x: box {64, 128}; map_wr: [E, H]
// box {64, E rounded up to 16}, halved when router_plan pairs the CTAs;
// map_ws: [1, H] box {64, 16} (used when the plan fuses the gate).
cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_wr, const CUtensorMap* map_ws, int T,
                          int H, int E, int k, const RouteSpec& spec, const void* x, const void* w_shared_gate,
                          int32_t* topk_idx, float* topk_w, float* shared_scale, uint32_t* err,
                          cudaStream_t stream);
// Launches of launch_router for these shapes.
int router_launches(int T, int H, int E, bool shared_gate);

// Decode-sized batches: routing and the permutation (counts, offsets, perm,
// inv, x_perm) in one single-CTA launch on the CUDA cores, when
// route_permute_is_tiny (T <= 8, E * H <= 128K router weights and T * H <=
// 48K: the batch's x rows fit the kernel's shared memory).
bool route_permute_is_tiny(int T, int H, int E, int k);
cudaError_t launch_route_permute_tiny(int T, int H, int E, int k, const RouteSpec& spec, const void* x,
                                      const void* w_router, const void* w_shared_gate, int32_t* topk_idx,
                                      float* topk_w, float* shared_scale, int32_t* counts, int32_t* offsets,
                                      int32_t* perm, int32_t* inv, void* x_perm, cudaStream_t stream);

// Permutation: bitmap build, scan, gather (see permute.cu); one launch for
// small batches (permute_is_small), which then uses no scratch.
size_t permute_scratch_bytes(int T, int E);
bool permute_is_small(int T, int E, int k);
int permute_launches(int T, int E, int k);
cudaError_t launch_permute(const int32_t* topk_idx, const void* x, int T, int H, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm, void* scratch,
                           uint32_t* err, cudaStream_t stream);

// How the SwiGLU GEMM loads its A tile (64 gate rows over the 64 up rows of
// the same features).  kStackedMap: one TMA box over a view whose extra
// dimension steps from the gate to the up weights (its stride is the distance
// between the two tensors); kTwoMaps: two 64-row boxes, one per tensor, used
// when that distance cannot be a TMA stride (it must be a non-zero multiple
// of 16 bytes below 2^40); one K block per stage.
enum SwiGLULoad { kStackedMap = 0, kTwoMaps = 1 };

// One operand set of the grouped GEMM: groups of rows of B against
// per-group weight blocks of A.
struct GemmSegment {
  const int32_t* offsets;  // [groups+1] device, or nullptr = one group of `rows` rows
  int groups;
  int rows;                // used when offsets == nullptr
  int nout;                // output features per group (multiple of 128)
  int K;                   // reduction length (multiple of 64)
  int bn;                  // token tile (16, 32, 64, 128, 256)
  void* out;               // [rows, ldo] bf16 (SwiGLU), fp32 / bf16 / fp16 (plain store)
  int ldo;
  int ksplit = 1;          // fp32 / fp16 store only: K cut into ksplit slices, slice s of
                           // the partial sums goes to out + s * slice_stride
  size_t slice_stride = 0; // elements
  int a_mode = kStackedMap;  // SwiGLU only
  int up_first = 0;          // SwiGLU, kStackedMap: the view's first plane is the up weights
  int gelu = 0;              // gated epilogue: GELU (erf form) instead of SiLU
};

// kEpiSwiGLU: gate and up rows stacked in one A tile, h = act(gate) * up in
// bf16 (act = SiLU, or GELU with GemmSegment::gelu).  kEpiStoreF32: one
// accumulator, fp32 out (K split allowed).  kEpiStoreBF16: one accumulator,
// bf16 out (the unfused gate / up projections of the fusion ablation).
// kEpiStoreF16: one accumulator, fp16 out (K split allowed; the down
// projection's expert outputs); a value beyond the fp16 range sets the device
// error word.
enum GemmEpilogue { kEpiSwiGLU = 0, kEpiStoreF32 = 1, kEpiStoreBF16 = 2, kEpiStoreF16 = 3 };

// How the grouped GEMM will run these segments: as CTA pairs (tcgen05
// cta_group::2; each CTA stages bn/2 token rows) or single CTAs, and with how
// many 64-wide K blocks per pipeline stage.  The maps must be built to match
// (token box bn/2 rows for a pair; box depth kps).
struct GemmPlan {
  bool pair;
  int kps;
  int nsub;  // sub-tiles per CTA and tile (1 or 2; see gemm_nsub)
};
// static_grid: the schedule ablation's plan (one 128-row weight tile per CTA,
// no CTA pairs), for launches with one CTA per tile.
GemmPlan grouped_gemm_plan(GemmEpilogue epi, int num_segments, const GemmSegment* segs, int num_sms,
                           bool static_grid = false);

// TMA descriptors of one grouped-GEMM segment.  The token rows [rows, K] are
// read through nb maps of increasing box height: b[i] brings (i + 1) * bstep
// rows (a 3-D view {64, rows, K/64} with box depth kps when kps > 1),
// nb * bstep = bn (bn/2 for a CTA pair; bstep = 16, or bn/8 above 128 rows),
// and every tile loads through the smallest box that covers its own rows, so
// no tile fetches rows it does not use beyond the next multiple of bstep.
//   Store:  a0 covers the [groups*nout, K] weights, box 128 rows.
//   SwiGLU, kStackedMap: a0 is the view {K, groups*nout, 2} (kps == 1) or
//           {64, groups*nout, 2, K/64} (kps > 1) of the gate and up weights
//           (plane stride = the distance between them), box 64 rows x 2
//           planes (x kps); one box per 64-feature sub-tile.
//   SwiGLU, kTwoMaps: a0 / a1 cover the gate / up weights, box 64 rows.
constexpr int kMaxBoxes = 8;
struct SegMaps {
  CUtensorMap a0, a1;
  CUtensorMap b[kMaxBoxes];
  int nb, bstep;
};

// Persistent grouped GEMM over one or two segments (seg_maps[s] for segment s).
// static_ctas > 0: the schedule ablation instead -- a grid of static_ctas
// CTAs (the tile count, known on the host), each running at most one tile,
// with the static_grid plan.
cudaError_t launch_grouped_gemm(GemmEpilogue epi, int num_segments, const GemmSegment* segs,
                                const SegMaps* seg_maps, int num_sms, uint32_t* err, cudaStream_t stream,
                                long long static_ctas = 0);

// Address of the current device's error word (nullptr if the device could
// not be set up).
uint32_t* device_error_word();

// h = act(g) * u elementwise over n bf16 values (n a multiple of 8; the
// unfused gated activation of the fusion ablation).
cudaError_t launch_gated_elementwise(const void* g, const void* u, void* h, size_t n, int gelu, cudaStream_t stream);

// Deterministic weighted combine of fp16 expert outputs.  y_perm (and
// y_shared) may hold nslices partial-sum slices slice_stride elements apart;
// they are added in slice order (fp32) before weighting.
cudaError_t launch_combine(const void* y_perm, const int32_t* inv, const float* topk_w, const void* y_shared,
                           const float* shared_scale, int T, int H, int k, void* out, cudaStream_t stream,
                           int nslices = 1, size_t slice_stride = 0, int nslices_shared = 1,
                           size_t slice_stride_shared = 0);

}  // namespace moe
