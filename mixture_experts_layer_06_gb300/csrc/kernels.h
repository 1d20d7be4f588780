// Host-side launchers of the MoE kernels (internal to the library).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

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

// Router GEMM (x [T,H] . W_r[E,H]^T on the tensor cores) fused with the score
// function and top-k.  map_x: box {64, 128}; map_wr: box {64, NE}, NE = E
// rounded up to 16.
cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_wr, int T, int H, int E, int k,
                          const RouteSpec& spec, int32_t* topk_idx, float* topk_w, uint32_t* err,
                          cudaStream_t stream);

// shared_scale[t] = sigmoid(x[t] . w_s)
cudaError_t launch_shared_gate(const void* x, const void* w_s, int T, int H, float* shared_scale,
                               cudaStream_t stream);

// Permutation: bitmap build, scan, gather (see permute.cu).
size_t permute_scratch_bytes(int T, int E);
cudaError_t launch_permute(const int32_t* topk_idx, const void* x, int T, int H, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm, void* scratch,
                           uint32_t* err, cudaStream_t stream);

// One operand set of the grouped GEMM: groups of rows of B against
// per-group weight blocks of A.
struct GemmSegment {
  const int32_t* offsets;  // [groups+1] device, or nullptr = one group of `rows` rows
  int groups;
  int rows;                // used when offsets == nullptr
  int nout;                // output features per group (multiple of 128)
  int K;                   // reduction length (multiple of 64)
  int bn;                  // token tile (16, 32, 64, 128, 256)
  void* out;               // [rows, ldo] bf16 (SwiGLU) or fp32 (plain store)
  int ldo;
};

enum GemmEpilogue { kEpiSwiGLU = 0, kEpiStoreF32 = 1 };

// Persistent grouped GEMM over one or two segments.  For segment s, A maps
// are [groups*nout, K] weights with box {64, 128}; B map is [rows, K] with
// box {64, bn}.  SwiGLU takes two A maps (gate, up) per segment.
cudaError_t launch_grouped_gemm(GemmEpilogue epi, int num_segments, const GemmSegment* segs,
                                const CUtensorMap* a0, const CUtensorMap* a1, const CUtensorMap* b,
                                int num_sms, uint32_t* err, cudaStream_t stream);

// Address of the current device's error word (nullptr if the device could
// not be set up).
uint32_t* device_error_word();

// Deterministic weighted combine.
cudaError_t launch_combine(const float* y_perm, const int32_t* inv, const float* topk_w, const float* y_shared,
                           const float* shared_scale, int T, int H, int k, void* out, cudaStream_t stream);

}  // namespace moe
