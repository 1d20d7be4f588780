// C ABI of the MoE layer forward: argument checks, TMA descriptors, workspace
// carve-up and the launch sequence.  Declarations and contracts: include/moe.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "kernels.h"
#include "ptx.cuh"

// Device error word (bit 0 timeout, bit 1 bounds, bits 8.. sites).
__device__ uint32_t g_moe_error_word;

std::atomic<unsigned long long> moe::g_launch_count{0};

// One thread waits on an mbarrier that nothing ever arrives on; the bounded
// wait must give up after limit_ns and record a timeout (failure-path check).
__global__ void selftest_wait_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    moe::mbar_init(&bar, 1);
    moe::fence_mbar_init();
    moe::mbar_wait_for(&bar, 0, limit_ns, err, moe::kSiteSelfTest);
  }
}

namespace {

using moe::GemmSegment;

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  uint32_t* err = nullptr;
  int num_sms = 0;
  void* ws = nullptr;  // moe_forward's cached workspace
  size_t ws_bytes = 0;
  cudaEvent_t ws_done = nullptr;  // recorded after the last moe_forward call's work
};

std::mutex g_mutex;
std::mutex g_ws_mutex;  // moe_forward's workspace: held while a call is enqueued
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

// Stage tracing (moe_set_trace_events).
constexpr int kTraceEvents = 6;
cudaEvent_t g_trace[kTraceEvents] = {};
bool g_trace_on = false;

void trace(int i, cudaStream_t s) {
  if (g_trace_on && g_trace[i] != nullptr) cudaEventRecord(g_trace[i], s);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Per-device constants, resolved once with that device current.
moe_status_t device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MOE_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_error_word) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    d.err = static_cast<uint32_t*>(p);
    d.ready = true;
  }
  *out = &d;
  return MOE_OK;
}

// bf16 [rows, cols] row-major, box {64 cols, box_rows rows}, 128-byte swizzle,
// out-of-range rows read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view {64, rows, cols/64} of a bf16 [rows, cols] row-major matrix, box
// {64, box_rows, box_k}: one request brings box_k consecutive 64-column
// blocks of box_rows rows, each block landing as its own 128-byte-swizzled
// tile.
bool make_map3d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_k) {
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, box_k};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weight / token-row map for the grouped GEMM: 2-D for one K block per
// stage, 3-D with box depth kps otherwise.
bool make_gemm_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, int kps) {
  return kps == 1 ? make_map(m, base, rows, cols, box_rows) : make_map3d(m, base, rows, cols, box_rows, kps);
}

// The token-row maps of a grouped-GEMM segment: boxes of bstep, 2 bstep, ...,
// max_rows rows (max_rows = the token tile per CTA: 16, 32, 64, 128 or 256;
// bstep = 16, or max_rows / 8 above 128).
bool make_token_maps(moe::SegMaps* m, const void* base, uint64_t rows, uint64_t cols, uint32_t max_rows, int kps) {
  m->bstep = static_cast<int>(max_rows > 16u * moe::kMaxBoxes ? max_rows / moe::kMaxBoxes : 16u);
  m->nb = static_cast<int>(max_rows) / m->bstep;
  if (m->nb < 1 || m->nb > moe::kMaxBoxes || static_cast<int>(max_rows) != m->nb * m->bstep) return false;
  for (int i = 0; i < m->nb; ++i)
    if (!make_gemm_map(&m->b[i], base, rows, cols, static_cast<uint32_t>((i + 1) * m->bstep), kps)) return false;
  return true;
}

// Stacked view of a SwiGLU segment's gate and up weights (both bf16
// [rows, K] row-major): one more dimension of extent 2 whose stride is the
// distance between the two tensors, lower address first, so that one box
// {64 columns, 64 rows, 2 planes} lands as 64 gate rows over the 64 up rows
// of the same features: one 128-row A tile.  With kps > 1 it is the 4-D view
// {64, rows, 2, K/64}, box depth kps (kps such tiles, one per K block).
// (A 5-D view that also spans consecutive 64-row blocks in one box measured
// far slower on GB300 than one 4-D box per block.)  Fails when the distance
// cannot be a TMA stride.
bool stackable(const void* w_gate, const void* w_up) {
  const uint64_t g = reinterpret_cast<uintptr_t>(w_gate), u = reinterpret_cast<uintptr_t>(w_up);
  const uint64_t dist = g < u ? u - g : g - u;
  return dist != 0 && dist % 16 == 0 && dist < (1ull << 40);
}

bool make_stacked_map(CUtensorMap* m, const void* w_gate, const void* w_up, uint64_t rows, uint64_t K, int kps,
                      int* up_first) {
  if (!stackable(w_gate, w_up)) return false;
  const uint64_t g = reinterpret_cast<uintptr_t>(w_gate), u = reinterpret_cast<uintptr_t>(w_up);
  *up_first = u < g ? 1 : 0;
  void* base = const_cast<void*>(u < g ? w_up : w_gate);
  const uint64_t dist = u < g ? g - u : u - g;
  if (kps == 1) {
    const cuuint64_t dims[3] = {K, rows, 2};
    const cuuint64_t strides[2] = {K * 2, dist};
    const cuuint32_t box[3] = {64, 64, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[4] = {64, rows, 2, K / 64};
  const cuuint64_t strides[3] = {K * 2, dist, 128};
  const cuuint32_t box[4] = {64, 64, 2, static_cast<cuuint32_t>(kps)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_dims(int T, int H, int F, int E, int k) {
  if (T < 0 || H <= 0 || F <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_VALUE;
  if (k > E || E > 256 || k > 16) return MOE_ERR_UNSUPPORTED;
  if (H % 128 != 0 || F % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t check_config(const moe_config_t& c, int H, int E, int k) {
  if (c.score != MOE_SCORE_SOFTMAX && c.score != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_VALUE;
  if (c.n_group > 1) {
    if (c.n_group > 16 || E % c.n_group != 0) return MOE_ERR_UNSUPPORTED;
    if (c.topk_group < 1 || c.topk_group > c.n_group) return MOE_ERR_INVALID_VALUE;
    if (c.group_topn < 1 || c.group_topn > 4 || c.group_topn > E / c.n_group) return MOE_ERR_UNSUPPORTED;
    if (k > c.topk_group * (E / c.n_group)) return MOE_ERR_INVALID_VALUE;
  }
  if (c.logit_bias != nullptr && !aligned16(c.logit_bias)) return MOE_ERR_INVALID_VALUE;
  if (c.F_shared < 0) return MOE_ERR_INVALID_VALUE;
  if (c.F_shared > 0) {
    if (c.F_shared % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!c.ws_gate || !c.ws_up || !c.ws_down) return MOE_ERR_INVALID_VALUE;
    if (!aligned16(c.ws_gate) || !aligned16(c.ws_up) || !aligned16(c.ws_down)) return MOE_ERR_INVALID_VALUE;
  }
  if (c.w_shared_gate != nullptr && !aligned16(c.w_shared_gate)) return MOE_ERR_INVALID_VALUE;
  if (c.activation != MOE_ACT_SILU && c.activation != MOE_ACT_GELU) return MOE_ERR_INVALID_VALUE;
  (void)H;
  return MOE_OK;
}

moe::RouteSpec route_spec(const moe_config_t& c) {
  moe::RouteSpec s{};
  s.sigmoid = c.score == MOE_SCORE_SIGMOID;
  s.renormalize = c.renormalize;
  s.route_scale = c.route_scale;
  s.n_group = c.n_group > 1 ? c.n_group : 1;
  s.topk_group = c.topk_group;
  s.group_topn = c.group_topn;
  s.logit_bias = c.logit_bias;
  return s;
}

// Token box of a routed segment (>= MOE_BOX_MIN_GROUPS experts): twice the
// power of two covering the mean rows per expert (at most 256).  The box
// bounds how many rows one tile can take, while every tile still runs MMAs of
// its own row count; with the mean as the box, the experts that routing
// leaves above the mean (about half of them even for uniform routing) split
// into two tiles that stream their weights twice.  Measured on GB300
// against the mean-sized box: Mixtral-shaped T=128 600 -> 482 us, T=512
// 598 -> 535 us; Qwen2-shaped T=512 891 -> 827 us; DeepSeek-V3-shaped T=2048
// 4152 -> 3844 us; skew T=512 alpha=0 268 -> 242 us, alpha=2 235 -> 172 us.
// A box of four times the mean helps heavy skew further but is slower where
// it moves the layer onto CTA pairs (Qwen2-shaped T=512, DeepSeek-V3-shaped
// T=2048) or where experts get a handful of rows (Mixtral-shaped T=32).  So
// experts averaging 32..63 rows take 4x (a 128-row box, still a single-CTA
// plan): skew T=512 alpha=2 (hot experts of ~500 rows) then runs half as many
// tiles.  A single group (dense or shared expert) keeps the exact box.
#ifndef MOE_BOX_SCALE
#define MOE_BOX_SCALE 2
#endif
#ifndef MOE_BOX_WIDE
#define MOE_BOX_WIDE 1
#endif
#ifndef MOE_BOX_MIN_GROUPS
#define MOE_BOX_MIN_GROUPS 2
#endif

// Token tile of the grouped GEMM: the smallest of 16..bn_max that covers the
// mean rows per group.
int choose_bn(long long rows, int groups, int bn_max = 256) {
  const long long avg = (rows + groups - 1) / (groups > 0 ? groups : 1);
  int bn = 16;
  while (bn < bn_max && bn < avg) bn <<= 1;
  if (groups >= MOE_BOX_MIN_GROUPS) {
    for (int i = 1; i < MOE_BOX_SCALE && bn < bn_max; i <<= 1) bn <<= 1;
    if (MOE_BOX_WIDE && bn == 64 && avg >= 32 && bn_max >= 128) bn = 128;
  }
  return bn;
}

// Router scratch: none (the K-split partial logits are reduced on chip).
size_t route_scratch(const moe_config_t& c, int T, int H, int E) {
  (void)c;
  (void)T;
  (void)H;
  (void)E;
  return 0;
}

// K-split of the down projection in moe_forward_ex.  When the routed rows
// give too few output tiles to fill the GPU several times over (small T:
// few active experts and one token tile each), K (= F) is cut into S <= 8
// slices whose partial sums go to separate fp16 y slices; the combine adds
// them in slice order, so the result stays deterministic.  S minimises a
// two-term estimate: the weight bytes times the wave-quantisation loss of
// tiles * S tiles on 152 SMs, plus the partial sums written and read back
// (2 * S * T k * H * 2 bytes); a slice keeps >= 8 K blocks.  The shared
// expert's K (= F_shared) is cut so that its slices are no longer than the
// routed ones.  Depends only on the shapes (not on the device), so that
// moe_workspace_bytes() can size the slices.
constexpr long long kTargetTiles = 6 * 152;
constexpr int kSms = 152;

struct Split {
  int routed = 1, shared = 1;
};

Split choose_split(const moe_config_t& c, int T, int H, int F, int E, int k) {
  Split sp;
  const long long Tk = static_cast<long long>(T) * k;
  const long long groups = Tk < E ? Tk : E;
  if (groups <= 0) return sp;
  const long long rows_per = (Tk + groups - 1) / groups;
  const int bn = choose_bn(Tk, E);
  const long long tiles = groups * (H / 128) * ((rows_per + bn - 1) / bn);
  const int kb = F / 64;
  if (tiles < kTargetTiles) {
    const double weights = 2.0 * groups * H * F;
    double best = 0.0;
    for (int S = 1; S <= 8 && kb / S >= 8; ++S) {
      const long long n = tiles * S;
      const double wave_loss = static_cast<double>((n + kSms - 1) / kSms * kSms) / static_cast<double>(n);
      const double cost = weights * wave_loss + 2.0 * S * Tk * H * 2.0;
      if (S == 1 || cost < best * 0.99) {  // a larger S must win by more than 1 %
        best = cost;
        sp.routed = S;
      }
    }
  }
  if (c.F_shared > 0) {
    const long long slice = F / sp.routed;
    const int kbs = c.F_shared / 64;
    while (sp.shared < 8 && c.F_shared / sp.shared > slice && kbs / (2 * sp.shared) >= 8) sp.shared <<= 1;
  }
  return sp;
}

// Token tile of a dense shared-expert segment that shares a launch with the
// routed segment: no larger than the routed tile (or 128), so that it does not
// force bigger stages and fewer accumulator slots on the routed tiles.
int shared_bn(long long rows, int routed_bn) { return choose_bn(rows, 1, routed_bn > 128 ? routed_bn : 128); }

// Workspace carve-up of moe_forward_ex, 256-byte aligned pieces.
struct Layout {
  size_t route_scratch, topk_idx, topk_w, shared_scale, counts, offsets, perm, inv, scratch, x_perm, h_perm, y_perm, h_shared,
      y_shared, total;
};

size_t up256(size_t v) { return (v + 255) & ~size_t(255); }

Layout layout(const moe_config_t& c, int T, int H, int F, int E, int k) {
  Layout L{};
  const size_t Tk = static_cast<size_t>(T) * k;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += up256(bytes);
    return at;
  };
  L.route_scratch = take(route_scratch(c, T, H, E));
  L.topk_idx = take(Tk * 4);
  L.topk_w = take(Tk * 4);
  L.shared_scale = take(static_cast<size_t>(T) * 4);
  L.counts = take(static_cast<size_t>(E) * 4);
  L.offsets = take(static_cast<size_t>(E + 1) * 4);
  L.perm = take(Tk * 4);
  L.inv = take(Tk * 4);
  L.scratch = take(moe::permute_scratch_bytes(T, E));
  L.x_perm = take(Tk * H * 2);
  L.h_perm = take(Tk * F * 2);
  const Split sp = choose_split(c, T, H, F, E, k);
  L.y_perm = take(sp.routed * Tk * H * 2);
  const size_t Fs = c.F_shared > 0 ? static_cast<size_t>(c.F_shared) : 0;
  L.h_shared = take(static_cast<size_t>(T) * Fs * 2);
  L.y_shared = take(Fs ? sp.shared * static_cast<size_t>(T) * H * 2 : 0);
  L.total = o;
  return L;
}

moe_status_t route_impl(DeviceState* d, const moe_config_t& c, const void* x, const void* w_router, int T, int H,
                        int E, int k, int32_t* topk_idx, float* topk_w, float* shared_scale, cudaStream_t stream) {
  CUtensorMap mx, mw, ms;
  const bool gate = c.w_shared_gate != nullptr && shared_scale != nullptr;
  const moe::RouterPlan plan = moe::router_plan(T, H, E, gate);
  const uint32_t wr_rows = (E + 15) / 16 * 16;
  if (!make_map(&mx, x, T, H, 128) || !make_map(&mw, w_router, E, H, plan.pair ? wr_rows / 2 : wr_rows))
    return MOE_ERR_CUDA;
  if (gate && !make_map(&ms, c.w_shared_gate, 1, H, 16)) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_router(mx, mw, gate ? &ms : nullptr, T, H, E, k, route_spec(c), x,
                                           gate ? c.w_shared_gate : nullptr, topk_idx, topk_w,
                                           gate ? shared_scale : nullptr, d->err, stream);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t permute_impl(DeviceState* d, const int32_t* topk_idx, const void* x, int T, int H, int E, int k,
                          int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm,
                          void* scratch, cudaStream_t stream) {
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), stream) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  return cuda_status(
      moe::launch_permute(topk_idx, x, T, H, E, k, counts, offsets, perm, inv, x_perm, scratch, d->err, stream));
}

// The two persistent GEMM launches (gate+up, then down) over the routed
// experts and, when given, the shared expert as a second segment.
struct FfnOperands {
  const void* x_rows;  // B of gate+up
  const int32_t* offsets;
  int rows, groups, H, F;
  const void *w_gate, *w_up, *w_down;
  void* h;
  void* y;         // fp16 [rows, H] (ksplit slices of rows*H)
  int ksplit = 1;  // down projection K slices
  int activation = MOE_ACT_SILU;
};

moe_status_t down_impl(DeviceState* d, int nseg, const FfnOperands* ops, cudaStream_t stream);

moe_status_t ffn_impl(DeviceState* d, int nseg, const FfnOperands* ops, cudaStream_t stream, bool traced = false) {
  moe::SegMaps maps[2];
  GemmSegment seg[2];
  // gate+up: B = token rows [rows, H], A = gate / up weights [groups*F, H]
  for (int s = 0; s < nseg; ++s) {
    const FfnOperands& o = ops[s];
    const int bn = (nseg > 1 && s == 1) ? shared_bn(o.rows, seg[0].bn) : choose_bn(o.rows, o.groups);
    seg[s] = GemmSegment{o.offsets, o.groups, o.rows, o.F, o.H, bn, o.h, o.F};
    seg[s].a_mode = stackable(o.w_gate, o.w_up) ? moe::kStackedMap : moe::kTwoMaps;
    seg[s].gelu = o.activation == MOE_ACT_GELU ? 1 : 0;
  }
  for (int attempt = 0;; ++attempt) {
    const moe::GemmPlan plan = moe::grouped_gemm_plan(moe::kEpiSwiGLU, nseg, seg, d->num_sms);
    bool replan = false;
    for (int s = 0; s < nseg && !replan; ++s) {
      const FfnOperands& o = ops[s];
      const uint64_t wrows = static_cast<uint64_t>(o.groups) * o.F;
      const uint32_t brows = plan.pair ? seg[s].bn / 2 : seg[s].bn;
      if (seg[s].a_mode == moe::kStackedMap) {
        if (!make_stacked_map(&maps[s].a0, o.w_gate, o.w_up, wrows, o.H, plan.kps, &seg[s].up_first)) {
          if (attempt > 0) return MOE_ERR_CUDA;
          seg[s].a_mode = moe::kTwoMaps;  // fall back to two boxes per stage
          replan = true;
          continue;
        }
        maps[s].a1 = maps[s].a0;
      } else if (!make_map(&maps[s].a0, o.w_gate, wrows, o.H, 64) || !make_map(&maps[s].a1, o.w_up, wrows, o.H, 64)) {
        return MOE_ERR_CUDA;
      }
      if (!make_token_maps(&maps[s], o.x_rows, o.rows, o.H, brows, plan.kps)) return MOE_ERR_CUDA;
    }
    if (!replan) break;
  }
  if (moe::launch_grouped_gemm(moe::kEpiSwiGLU, nseg, seg, maps, d->num_sms, d->err, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (traced) trace(3, stream);
  return down_impl(d, nseg, ops, stream);
}

// The down projection: B = h [rows, F], A = down weights [groups*H, F], fp16 y
// (K-split slices when ops ask for them).
moe_status_t down_impl(DeviceState* d, int nseg, const FfnOperands* ops, cudaStream_t stream) {
  moe::SegMaps maps[2];
  GemmSegment seg[2];
  for (int s = 0; s < nseg; ++s) {
    const FfnOperands& o = ops[s];
    const int bn = (nseg > 1 && s == 1) ? shared_bn(o.rows, choose_bn(ops[0].rows, ops[0].groups))
                                        : choose_bn(o.rows, o.groups);
    seg[s] = GemmSegment{o.offsets, o.groups, o.rows, o.H, o.F, bn, o.y, o.H, o.ksplit,
                         static_cast<size_t>(o.rows) * o.H};
  }
  const moe::GemmPlan plan = moe::grouped_gemm_plan(moe::kEpiStoreF16, nseg, seg, d->num_sms);
  for (int s = 0; s < nseg; ++s) {
    const FfnOperands& o = ops[s];
    const uint64_t wrows = static_cast<uint64_t>(o.groups) * o.H;
    const uint32_t brows = plan.pair ? seg[s].bn / 2 : seg[s].bn;
    if (!make_gemm_map(&maps[s].a0, o.w_down, wrows, o.F, 128, plan.kps) ||
        !make_token_maps(&maps[s], o.h, o.rows, o.F, brows, plan.kps))
      return MOE_ERR_CUDA;
    maps[s].a1 = maps[s].a0;
  }
  if (moe::launch_grouped_gemm(moe::kEpiStoreF16, nseg, seg, maps, d->num_sms, d->err, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Fusion ablation: gate and up as two grouped GEMMs with bf16 outputs in
// global memory, the gated activation as an element-wise pass, then the
// same down projection.
moe_status_t ffn_unfused_impl(DeviceState* d, const FfnOperands& o, void* g, void* u, cudaStream_t stream) {
  GemmSegment seg = GemmSegment{o.offsets, o.groups, o.rows, o.F, o.H, choose_bn(o.rows, o.groups), g, o.F};
  const moe::GemmPlan plan = moe::grouped_gemm_plan(moe::kEpiStoreBF16, 1, &seg, d->num_sms);
  const uint64_t wrows = static_cast<uint64_t>(o.groups) * o.F;
  const uint32_t brows = plan.pair ? seg.bn / 2 : seg.bn;
  moe::SegMaps maps;
  if (!make_token_maps(&maps, o.x_rows, o.rows, o.H, brows, plan.kps)) return MOE_ERR_CUDA;
  const void* w[2] = {o.w_gate, o.w_up};
  void* dst[2] = {g, u};
  for (int i = 0; i < 2; ++i) {
    if (!make_gemm_map(&maps.a0, w[i], wrows, o.H, 128, plan.kps)) return MOE_ERR_CUDA;
    maps.a1 = maps.a0;
    seg.out = dst[i];
    if (moe::launch_grouped_gemm(moe::kEpiStoreBF16, 1, &seg, &maps, d->num_sms, d->err, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (moe::launch_gated_elementwise(g, u, o.h, static_cast<size_t>(o.rows) * o.F, o.activation == MOE_ACT_GELU,
                                    stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return down_impl(d, 1, &o, stream);
}

// Schedule ablation: the expert counts are read back to the host (a
// synchronisation), the token tile is a fixed block_m, and each grouped GEMM
// is launched with one CTA per tile, one 128-row weight tile per CTA.
moe_status_t ffn_static_impl(DeviceState* d, const FfnOperands& o, int block_m, cudaStream_t stream) {
  std::vector<int32_t> off(static_cast<size_t>(o.groups) + 1);
  if (cudaMemcpyAsync(off.data(), o.offsets, off.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  long long token_tiles = 0;
  for (int g = 0; g < o.groups; ++g) {
    const long long r = static_cast<long long>(off[g + 1]) - off[g];
    if (r < 0 || off[g + 1] > o.rows) return MOE_ERR_INVALID_VALUE;
    token_tiles += (r + block_m - 1) / block_m;
  }
  if (token_tiles == 0) return MOE_OK;
  // gate+up: 64 features per CTA (one stacked gate/up tile)
  GemmSegment seg = GemmSegment{o.offsets, o.groups, o.rows, o.F, o.H, block_m, o.h, o.F};
  seg.a_mode = stackable(o.w_gate, o.w_up) ? moe::kStackedMap : moe::kTwoMaps;
  seg.gelu = o.activation == MOE_ACT_GELU ? 1 : 0;
  moe::SegMaps maps;
  for (int attempt = 0;; ++attempt) {
    const moe::GemmPlan plan = moe::grouped_gemm_plan(moe::kEpiSwiGLU, 1, &seg, d->num_sms, true);
    const uint64_t wrows = static_cast<uint64_t>(o.groups) * o.F;
    if (seg.a_mode == moe::kStackedMap) {
      if (!make_stacked_map(&maps.a0, o.w_gate, o.w_up, wrows, o.H, plan.kps, &seg.up_first)) {
        if (attempt > 0) return MOE_ERR_CUDA;
        seg.a_mode = moe::kTwoMaps;
        continue;
      }
      maps.a1 = maps.a0;
    } else if (!make_map(&maps.a0, o.w_gate, wrows, o.H, 64) || !make_map(&maps.a1, o.w_up, wrows, o.H, 64)) {
      return MOE_ERR_CUDA;
    }
    if (!make_token_maps(&maps, o.x_rows, o.rows, o.H, block_m, plan.kps)) return MOE_ERR_CUDA;
    break;
  }
  if (moe::launch_grouped_gemm(moe::kEpiSwiGLU, 1, &seg, &maps, d->num_sms, d->err, stream,
                               token_tiles * (o.F / 64)) != cudaSuccess)
    return MOE_ERR_CUDA;
  // down: 128 output rows per CTA
  GemmSegment dseg = GemmSegment{o.offsets, o.groups, o.rows, o.H, o.F, block_m, o.y, o.H, 1,
                                 static_cast<size_t>(o.rows) * o.H};
  const moe::GemmPlan dplan = moe::grouped_gemm_plan(moe::kEpiStoreF16, 1, &dseg, d->num_sms, true);
  moe::SegMaps dmaps;
  if (!make_gemm_map(&dmaps.a0, o.w_down, static_cast<uint64_t>(o.groups) * o.H, o.F, 128, dplan.kps) ||
      !make_token_maps(&dmaps, o.h, o.rows, o.F, block_m, dplan.kps))
    return MOE_ERR_CUDA;
  dmaps.a1 = dmaps.a0;
  if (moe::launch_grouped_gemm(moe::kEpiStoreF16, 1, &dseg, &dmaps, d->num_sms, d->err, stream,
                               token_tiles * (o.H / 128)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Kernels moe_forward_ex launches for these shapes (its launch sequence below).
int forward_launches(const moe_config_t& c, int T, int H, int E, int k) {
  if (T == 0) return 0;
  const bool tiny = moe::route_permute_is_tiny(T, H, E, k);
  const int route = tiny ? 1 : moe::router_launches(T, H, E, c.w_shared_gate != nullptr);
  const int permute = tiny ? 0 : moe::permute_launches(T, E, k);
  const int ffn = 2;
  const int combine = 1;
  return route + permute + ffn + combine;
}

}  // namespace

namespace moe {
uint32_t* device_error_word() {
  DeviceState* d = nullptr;
  return device_state(&d) == MOE_OK ? d->err : nullptr;
}
}  // namespace moe

extern "C" {

void moe_config_default(moe_config_t* cfg) {
  if (cfg == nullptr) return;
  std::memset(cfg, 0, sizeof(*cfg));
  cfg->score = MOE_SCORE_SOFTMAX;
  cfg->renormalize = 1;
  cfg->route_scale = 1.0f;
  cfg->n_group = 1;
  cfg->topk_group = 1;
  cfg->group_topn = 0;
  cfg->activation = MOE_ACT_SILU;
}

int moe_abi_version(void) { return 102; }

moe_status_t moe_set_trace_events(void* const* events, int count) {
  if (events == nullptr || count == 0) {
    g_trace_on = false;
    return MOE_OK;
  }
  if (count != kTraceEvents) return MOE_ERR_INVALID_VALUE;
  bool any = false;
  for (int i = 0; i < kTraceEvents; ++i) any = any || events[i] != nullptr;
  if (!any) return MOE_ERR_INVALID_VALUE;
  for (int i = 0; i < kTraceEvents; ++i) g_trace[i] = static_cast<cudaEvent_t>(events[i]);
  g_trace_on = true;
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_VALUE: return "MOE_ERR_INVALID_VALUE";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
  }
  return "MOE_ERR_UNKNOWN";
}

size_t moe_route_scratch_bytes(const moe_config_t* cfg, int T, int H, int E) {
  moe_config_t c;
  if (cfg)
    c = *cfg;
  else
    moe_config_default(&c);
  if (T < 0 || H <= 0 || H % 128 != 0 || E <= 0 || E > 256) return 0;
  return route_scratch(c, T, H, E);
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router, int T, int H, int E, int k,
                       int32_t* topk_idx, float* topk_w, float* shared_scale, void* scratch, size_t scratch_bytes,
                       moe_stream_t stream) {
  moe_config_t c;
  if (cfg)
    c = *cfg;
  else
    moe_config_default(&c);
  moe_status_t st = check_dims(T, H, 128, E, k);
  if (st != MOE_OK) return st;
  if ((st = check_config(c, H, E, k)) != MOE_OK) return st;
  if (!x || !w_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_VALUE;
  if (c.w_shared_gate && !shared_scale) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_INVALID_VALUE;
  if (T == 0) return MOE_OK;
  const size_t need = route_scratch(c, T, H, E);
  if (need > 0 && (!scratch || !aligned16(scratch))) return MOE_ERR_INVALID_VALUE;
  if (scratch_bytes < need) return MOE_ERR_WORKSPACE;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != MOE_OK) return st;
  return route_impl(d, c, x, w_router, T, H, E, k, topk_idx, topk_w, shared_scale,
                    reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_permute_scratch_bytes(int T, int E) {
  if (T < 0 || E <= 0) return 0;
  return moe::permute_scratch_bytes(T, E);
}

moe_status_t moe_permute(const int32_t* topk_idx, const void* x, int T, int H, int E, int k, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm, void* scratch,
                         size_t scratch_bytes, moe_stream_t stream) {
  moe_status_t st = check_dims(T, H, 128, E, k);
  if (st != MOE_OK) return st;
  if (!counts || !offsets) return MOE_ERR_INVALID_VALUE;
  if (T > 0 && (!topk_idx || !x || !perm || !inv || !x_perm || !scratch)) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(x) || !aligned16(x_perm) || !aligned16(scratch)) return MOE_ERR_INVALID_VALUE;
  if (T > 0 && scratch_bytes < moe::permute_scratch_bytes(T, E)) return MOE_ERR_WORKSPACE;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != MOE_OK) return st;
  return permute_impl(d, topk_idx, x, T, H, E, k, counts, offsets, perm, inv, x_perm, scratch,
                      reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn(const void* x_perm, const int32_t* offsets, int rows, int H, int F, int E,
                            const void* w_gate, const void* w_up, const void* w_down, void* h, void* y,
                            moe_stream_t stream) {
  return moe_expert_ffn_ex(x_perm, offsets, rows, H, F, E, w_gate, w_up, w_down, MOE_ACT_SILU, h, y, stream);
}

moe_status_t moe_expert_ffn_static(const void* x_perm, const int32_t* offsets, int rows, int H, int F, int E,
                                   const void* w_gate, const void* w_up, const void* w_down, int block_m, void* h,
                                   void* y, moe_stream_t stream) {
  if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128 && block_m != 256)
    return MOE_ERR_INVALID_VALUE;
  moe_status_t st = check_dims(rows, H, F, E, 1);
  if (st != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  if (!x_perm || !offsets || !w_gate || !w_up || !w_down || !h || !y) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(h) ||
      !aligned16(y))
    return MOE_ERR_INVALID_VALUE;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != MOE_OK) return st;
  FfnOperands o{x_perm, offsets, rows, E, H, F, w_gate, w_up, w_down, h, y};
  return ffn_static_impl(d, o, block_m, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn_unfused(const void* x_perm, const int32_t* offsets, int rows, int H, int F, int E,
                                    const void* w_gate, const void* w_up, const void* w_down, int activation,
                                    void* g, void* u, void* h, void* y, moe_stream_t stream) {
  if (activation != MOE_ACT_SILU && activation != MOE_ACT_GELU) return MOE_ERR_INVALID_VALUE;
  moe_status_t st = check_dims(rows, H, F, E, 1);
  if (st != MOE_OK) return st;
  if (offsets == nullptr && E != 1) return MOE_ERR_INVALID_VALUE;
  if (rows == 0) return MOE_OK;
  if (!x_perm || !w_gate || !w_up || !w_down || !g || !u || !h || !y) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(g) ||
      !aligned16(u) || !aligned16(h) || !aligned16(y))
    return MOE_ERR_INVALID_VALUE;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != MOE_OK) return st;
  FfnOperands o{x_perm, offsets, rows, E, H, F, w_gate, w_up, w_down, h, y};
  o.activation = activation;
  return ffn_unfused_impl(d, o, g, u, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn_ex(const void* x_perm, const int32_t* offsets, int rows, int H, int F, int E,
                               const void* w_gate, const void* w_up, const void* w_down, int activation, void* h,
                               void* y, moe_stream_t stream) {
  if (activation != MOE_ACT_SILU && activation != MOE_ACT_GELU) return MOE_ERR_INVALID_VALUE;
  moe_status_t st = check_dims(rows, H, F, E, 1);
  if (st != MOE_OK) return st;
  if (offsets == nullptr && E != 1) return MOE_ERR_INVALID_VALUE;
  if (rows == 0) return MOE_OK;
  if (!x_perm || !w_gate || !w_up || !w_down || !h || !y) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(x_perm) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(h) ||
      !aligned16(y))
    return MOE_ERR_INVALID_VALUE;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != MOE_OK) return st;
  FfnOperands o{x_perm, offsets, rows, E, H, F, w_gate, w_up, w_down, h, y};
  o.activation = activation;
  return ffn_impl(d, 1, &o, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const void* y_perm, const int32_t* inv, const float* topk_w, const void* y_shared,
                         const float* shared_scale, int T, int H, int k, void* out, moe_stream_t stream) {
  if (T < 0 || H <= 0 || k <= 0 || k > 16) return MOE_ERR_INVALID_VALUE;
  if (H % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_perm || !inv || !topk_w || !out) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(y_perm) || !aligned16(out) || !aligned16(y_shared)) return MOE_ERR_INVALID_VALUE;
  return cuda_status(moe::launch_combine(y_perm, inv, topk_w, y_shared, shared_scale, T, H, k, out,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_workspace_bytes(const moe_config_t* cfg, int T, int H, int F, int E, int k) {
  moe_config_t c;
  if (cfg)
    c = *cfg;
  else
    moe_config_default(&c);
  if (check_dims(T, H, F, E, k) != MOE_OK) return 0;
  return layout(c, T, H, F, E, k).total;
}

moe_status_t moe_forward_ex(const moe_config_t* cfg, const void* x, const void* w_router, const void* w_gate,
                            const void* w_up, const void* w_down, int T, int H, int F, int E, int k, void* out,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  moe_config_t c;
  if (cfg)
    c = *cfg;
  else
    moe_config_default(&c);
  moe_status_t st = check_dims(T, H, F, E, k);
  if (st != MOE_OK) return st;
  if ((st = check_config(c, H, E, k)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !w_gate || !w_up || !w_down || !out || !workspace) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_INVALID_VALUE;
  const Layout L = layout(c, T, H, F, E, k);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto at = [&](size_t off) { return static_cast<void*>(ws + off); };
  int32_t* topk_idx = static_cast<int32_t*>(at(L.topk_idx));
  float* topk_w = static_cast<float*>(at(L.topk_w));
  float* shared_scale = c.w_shared_gate ? static_cast<float*>(at(L.shared_scale)) : nullptr;
  int32_t* offsets = static_cast<int32_t*>(at(L.offsets));
  int32_t* inv = static_cast<int32_t*>(at(L.inv));
  const int Tk = T * k;

  trace(0, s);
  if (moe::route_permute_is_tiny(T, H, E, k)) {
    // decode-sized batch: routing and grouping in one launch (the permute stage is empty)
    if (moe::launch_route_permute_tiny(T, H, E, k, route_spec(c), x, w_router, c.w_shared_gate, topk_idx, topk_w,
                                       shared_scale, static_cast<int32_t*>(at(L.counts)), offsets,
                                       static_cast<int32_t*>(at(L.perm)), inv, at(L.x_perm), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    trace(1, s);
  } else {
    if ((st = route_impl(d, c, x, w_router, T, H, E, k, topk_idx, topk_w, shared_scale, s)) != MOE_OK) return st;
    trace(1, s);
    if ((st = permute_impl(d, topk_idx, x, T, H, E, k, static_cast<int32_t*>(at(L.counts)), offsets,
                           static_cast<int32_t*>(at(L.perm)), inv, at(L.x_perm), at(L.scratch), s)) != MOE_OK)
      return st;
  }
  const Split sp = choose_split(c, T, H, F, E, k);
  FfnOperands ops[2];
  ops[0] = FfnOperands{at(L.x_perm), offsets, Tk, E, H, F, w_gate, w_up, w_down, at(L.h_perm),
                       at(L.y_perm), sp.routed, c.activation};
  int nseg = 1;
  void* y_shared = nullptr;
  if (c.F_shared > 0) {
    y_shared = at(L.y_shared);
    ops[1] = FfnOperands{x, nullptr, T, 1, H, c.F_shared, c.ws_gate, c.ws_up, c.ws_down, at(L.h_shared), y_shared,
                         sp.shared, c.activation};
    nseg = 2;
  }
  trace(2, s);
  if ((st = ffn_impl(d, nseg, ops, s, true)) != MOE_OK) return st;
  trace(4, s);
  st = cuda_status(moe::launch_combine(at(L.y_perm), inv, topk_w, y_shared, shared_scale, T,
                                       H, k, out, s, sp.routed, static_cast<size_t>(Tk) * H, sp.shared,
                                       static_cast<size_t>(T) * H));
  trace(5, s);
  return st;
}

moe_status_t moe_forward(const void* x, const void* w_router, const void* w_gate, const void* w_up,
                         const void* w_down, int T, int H, int F, int E, int k, void* out, moe_stream_t stream) {
  moe_config_t c;
  moe_config_default(&c);
  moe_status_t st = check_dims(T, H, F, E, k);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  // the pointer checks of moe_forward_ex, before the workspace is grown
  if (!x || !w_router || !w_gate || !w_up || !w_down || !out) return MOE_ERR_INVALID_VALUE;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
      !aligned16(out))
    return MOE_ERR_INVALID_VALUE;
  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != MOE_OK) return st;
  const size_t need = layout(c, T, H, F, E, k).total;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return MOE_ERR_UNSUPPORTED;  // moe_forward_ex is the capturable form
  // Calls are ordered through ws_done: each call's work waits for the previous
  // call's work (on whatever stream it ran), so the one workspace is never
  // used by two calls at once and is never freed under a call still running.
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  if (d->ws_done == nullptr && cudaEventCreateWithFlags(&d->ws_done, cudaEventDisableTiming) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamWaitEvent(s, d->ws_done, 0) != cudaSuccess) return MOE_ERR_CUDA;
  if (d->ws_bytes < need) {
    if (d->ws != nullptr && cudaFreeAsync(d->ws, s) != cudaSuccess) return MOE_ERR_CUDA;
    d->ws = nullptr;
    d->ws_bytes = 0;
    if (cudaMallocAsync(&d->ws, need, s) != cudaSuccess) return MOE_ERR_CUDA;
    d->ws_bytes = need;
  }
  st = moe_forward_ex(&c, x, w_router, w_gate, w_up, w_down, T, H, F, E, k, out, d->ws, need, stream);
  if (cudaEventRecord(d->ws_done, s) != cudaSuccess && st == MOE_OK) st = MOE_ERR_CUDA;
  return st;
}

int moe_forward_launches(const moe_config_t* cfg, int T, int H, int F, int E, int k) {
  moe_config_t c;
  if (cfg)
    c = *cfg;
  else
    moe_config_default(&c);
  if (check_dims(T, H, F, E, k) != MOE_OK || check_config(c, H, E, k) != MOE_OK) return -1;
  return forward_launches(c, T, H, E, k);
}

unsigned long long moe_launches_issued(void) { return moe::g_launch_count.load(std::memory_order_relaxed); }

moe_status_t moe_selftest_wait_timeout(uint32_t limit_us, moe_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return MOE_ERR_INVALID_VALUE;
  DeviceState* d = nullptr;
  moe_status_t st = device_state(&d);
  if (st != MOE_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(uint64_t(limit_us) * 1000u, d->err);
  return cuda_status(cudaGetLastError());
}

moe_status_t moe_device_error(moe_stream_t stream, uint32_t* raw) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_moe_error_word, sizeof(w)) != cudaSuccess) return MOE_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_moe_error_word, &zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_CUDA;
  if (raw) *raw = w;
  if (w & moe::kErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (w & moe::kErrBounds) return MOE_ERR_DEVICE_BOUNDS;
  return MOE_OK;
}

}  // extern "C"
