// Token permutation onto experts.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "The reading":
// after scoring, the tokens are reordered onto experts so that each expert's
// rows are contiguous for a variable-size GEMM.  The order inside an expert is
// the token order (a stable counting sort by expert id).
//
// Instead of atomics, the sort is built from per-expert token bitmaps:
//   bitmap[w][e] bit b  <=> token 32*w + b picked expert e
//   rank of (t, e)      =  offsets[e] + sum_{w' < w} popc(bitmap[w'][e])
//                          + popc(bitmap[w][e] & lanes below b)
// which is deterministic and stable by construction.  Three launches:
//   1. bitmap_kernel: one warp per 32 tokens, __match_any_sync groups lanes by
//      expert, one word per (word, expert) written, coalesced;
//   2. scan_kernel: one CTA; per-expert popcount prefix over words, counts,
//      offsets (exclusive scan), and rowbase[w][e] = first grouped row of word w;
//   3. gather_kernel: one warp per token computes its k grouped rows, writes
//      perm / inv and copies x[t] into those rows with 16-byte vectors.
#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;

__global__ void bitmap_kernel(const int32_t* __restrict__ idx, int T, int E, int k, int W,
                              uint32_t* __restrict__ bitmap, uint32_t* err) {
  __shared__ uint32_t words[kWarpsPerBlock][256];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarpsPerBlock + warp;
  if (w >= W) return;  // warp-uniform
  uint32_t* mine = words[warp];
  for (int e = lane; e < E; e += 32) mine[e] = 0;
  __syncwarp();
  const int t = w * 32 + lane;
  for (int j = 0; j < k; ++j) {
    int e = -1;
    if (t < T) {
      e = idx[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) {
        raise_error(err, kErrBounds, kSitePermuteIndex);
        e = -1;
      }
    }
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) {
      if (mine[e] & peers) raise_error(err, kErrBounds, kSitePermuteIndex);  // expert repeated in a token
      mine[e] |= peers;
    }
    __syncwarp();
  }
  for (int e = lane; e < E; e += 32) bitmap[static_cast<size_t>(w) * E + e] = mine[e];
}

__global__ void __launch_bounds__(1024, 1)
    scan_kernel(const uint32_t* __restrict__ bitmap, int W, int E, int32_t* __restrict__ counts,
                int32_t* __restrict__ offsets, uint32_t* __restrict__ rowbase) {
  __shared__ uint32_t partial[1024];
  __shared__ int32_t off_s[257];
  __shared__ int32_t warp_tot[8];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int nc = 1024 / E;  // chunks of words per expert
  const int e = tid % E, c = tid / E;
  const bool active = c < nc;
  const int L = (W + nc - 1) / nc;
  const int w0 = c * L, w1 = min(W, w0 + L);

  uint32_t sum = 0;
  if (active)
    for (int w = w0; w < w1; ++w) sum += __popc(bitmap[static_cast<size_t>(w) * E + e]);
  partial[tid] = sum;
  __syncthreads();
  if (tid < E) {
    uint32_t run = 0;
    for (int cc = 0; cc < nc; ++cc) {
      const uint32_t v = partial[cc * E + tid];
      partial[cc * E + tid] = run;
      run += v;
    }
    counts[tid] = static_cast<int32_t>(run);
    off_s[tid] = static_cast<int32_t>(run);
  }
  __syncthreads();
  // Exclusive scan of the E <= 256 counts by the first 8 warps: shuffle scan
  // inside each warp, then the warp totals.
  int32_t cnt = 0, incl = 0;
  if (tid < 256) {
    cnt = tid < E ? off_s[tid] : 0;
    incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if ((tid & 31) >= o) incl += n;
    }
    if ((tid & 31) == 31) warp_tot[tid >> 5] = incl;
  }
  __syncthreads();
  if (tid < 256) {
    int32_t base = 0;
    for (int w = 0; w < (tid >> 5); ++w) base += warp_tot[w];
    if (tid < E) off_s[tid] = base + incl - cnt;
    if (tid == E - 1) off_s[E] = base + incl;
  }
  __syncthreads();
  for (int ee = tid; ee <= E; ee += 1024) offsets[ee] = off_s[ee];
  if (active) {
    uint32_t run = static_cast<uint32_t>(off_s[e]) + partial[tid];
    for (int w = w0; w < w1; ++w) {
      rowbase[static_cast<size_t>(w) * E + e] = run;
      run += __popc(bitmap[static_cast<size_t>(w) * E + e]);
    }
  }
}

// Grid (token blocks of 8, chunks of 256 columns): warp = (token, chunk).
// Every warp computes its token's k grouped rows; the chunk-0 warp writes
// perm / inv; each warp copies its 512-byte piece of x[t] to the k rows.
__global__ void gather_kernel(const int32_t* __restrict__ idx, const uint4* __restrict__ x, int T, int H8, int E,
                              int k, const uint32_t* __restrict__ bitmap, const uint32_t* __restrict__ rowbase,
                              int32_t* __restrict__ perm, int32_t* __restrict__ inv, uint4* __restrict__ x_perm,
                              uint32_t* err) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;  // warp-uniform
  const int rows = T * k;
  int r = -1;
  if (lane < k) {
    const int e = idx[static_cast<size_t>(t) * k + lane];
    if (e >= 0 && e < E) {
      const size_t we = static_cast<size_t>(t >> 5) * E + e;
      r = static_cast<int>(rowbase[we] + __popc(bitmap[we] & ((1u << (t & 31)) - 1u)));
      if (r >= rows) {
        if (blockIdx.y == 0) raise_error(err, kErrBounds, kSitePermuteIndex);
        r = -1;
      }
    }
    if (blockIdx.y == 0) {
      if (r >= 0) perm[r] = t * k + lane;
      inv[static_cast<size_t>(t) * k + lane] = r;
    }
  }
  const int v = blockIdx.y * 32 + lane;
  const bool active = v < H8;
  uint4 val = make_uint4(0, 0, 0, 0);
  if (active) val = x[static_cast<size_t>(t) * H8 + v];
  for (int j = 0; j < k; ++j) {
    const int rj = __shfl_sync(0xFFFFFFFFu, r, j);  // all lanes take part
    if (active && rj >= 0) x_perm[static_cast<size_t>(rj) * H8 + v] = val;
  }
}

// Small batches (T <= kSmallT): the whole permutation in one launch.  Every
// CTA builds the token bitmaps, the counts, the exclusive scan and the row
// bases of all T tokens in its own shared memory (at most kSmallT / 32 * E
// words each: cheap to repeat), then copies its share of the x_perm rows;
// CTA 0 also writes counts, offsets, perm and inv.
// Same arithmetic, same results as the three-launch form.
constexpr int kSmallT = 512;
constexpr int kSmallThreads = 256;
constexpr int kSmallIdx = 2048;  // most copies (T * k) a one-launch permute takes
constexpr int kSmallMaxK = 16;   // most experts per token

__global__ void __launch_bounds__(kSmallThreads)
    permute_small_kernel(const int32_t* __restrict__ idx, const uint4* __restrict__ x, int T, int H8, int E, int k,
                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                         int32_t* __restrict__ inv, uint4* __restrict__ x_perm, uint32_t* err) {
  __shared__ uint32_t bm[kSmallT / 32][256];
  __shared__ uint32_t rowbase[kSmallT / 32][256];
  __shared__ int32_t off_s[257];
  __shared__ int32_t warp_tot[8];
  __shared__ int32_t idx_s[kSmallIdx];  // the expert ids (-1: out of range), for the row lookups
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int W = (T + 31) / 32;
  for (int i = tid; i < W * 256; i += kSmallThreads) bm[i / 256][i % 256] = 0;
  __syncthreads();
  // bitmaps: warp w' handles token words w', w' + 8, ...; a token's k ids are
  // loaded together (one round trip, not k)
  for (int w = warp; w < W; w += kSmallThreads / 32) {
    const int t = w * 32 + lane;
    int ev[kSmallMaxK];
#pragma unroll
    for (int j = 0; j < kSmallMaxK; ++j) ev[j] = (j < k && t < T) ? idx[static_cast<size_t>(t) * k + j] : -1;
#pragma unroll
    for (int j = 0; j < kSmallMaxK; ++j) {
      if (j >= k) break;  // uniform
      int e = ev[j];
      if (t < T) {
        if (e < 0 || e >= E) {
          if (blockIdx.x == 0) raise_error(err, kErrBounds, kSitePermuteIndex);
          e = -1;
        }
        idx_s[t * k + j] = e;
      }
      const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) {
        if ((bm[w][e] & peers) && blockIdx.x == 0) raise_error(err, kErrBounds, kSitePermuteIndex);
        bm[w][e] |= peers;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // counts and the exclusive scan (thread e < E <= 256)
  int32_t cnt = 0;
  if (tid < E)
    for (int w = 0; w < W; ++w) cnt += __popc(bm[w][tid]);
  int32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int32_t base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  if (tid < E) {
    off_s[tid] = base + incl - cnt;
    uint32_t run = static_cast<uint32_t>(base + incl - cnt);
    for (int w = 0; w < W; ++w) {
      rowbase[w][tid] = run;
      run += __popc(bm[w][tid]);
    }
    if (blockIdx.x == 0) counts[tid] = cnt;
  }
  if (tid == E - 1) off_s[E] = base + incl;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = tid; e <= E; e += kSmallThreads) offsets[e] = off_s[e];
  // grouped row of copy q = t * k + j (-1: dropped id)
  const int rows = T * k;
  auto row_of = [&](int q) {
    const int t = q / k;
    const int e = idx_s[q];
    if (e < 0) return -1;
    const int r = static_cast<int>(rowbase[t >> 5][e] + __popc(bm[t >> 5][e] & ((1u << (t & 31)) - 1u)));
    return r < rows ? r : -1;
  };
  if (blockIdx.x == 0)
    for (int q = tid; q < rows; q += kSmallThreads) {
      const int r = row_of(q);
      if (r >= 0) perm[r] = q;
      inv[q] = r;
    }
  // x_perm: CTA b copies the rows of copies b, b + gridDim.x, ... in 16-byte
  // pieces, four loads in flight per thread
  for (int q = blockIdx.x; q < rows; q += gridDim.x) {
    const int r = row_of(q);  // the same for every thread of the CTA
    if (r < 0) continue;
    const uint4* src = x + static_cast<size_t>(q / k) * H8;
    uint4* dst = x_perm + static_cast<size_t>(r) * H8;
    for (int v0 = tid; v0 < H8; v0 += 4 * kSmallThreads) {
      uint4 val[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + u * kSmallThreads < H8) val[u] = src[v0 + u * kSmallThreads];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + u * kSmallThreads < H8) dst[v0 + u * kSmallThreads] = val[u];
    }
  }
}

}  // namespace

// The one-launch form repeats the bitmap work in every CTA and copies with
// fewer threads in flight: measured on GB300 it wins up to about 2048 grouped
// rows (Mixtral-shaped T=512: 10.5 vs 14 us) and loses above (4096 rows:
// 29-35 vs 17-21 us).
constexpr int kSmallRows = 2048;
static_assert(kSmallRows <= kSmallIdx, "the one-launch permute keeps every copy's expert id in shared memory");

bool permute_is_small(int T, int E, int k) { return T <= kSmallT && E <= 256 && T * k <= kSmallRows; }

int permute_launches(int T, int E, int k) { return T == 0 ? 0 : permute_is_small(T, E, k) ? 1 : 3; }

size_t permute_scratch_bytes(int T, int E) {
  const size_t W = (static_cast<size_t>(T) + 31) / 32;
  return 2 * W * static_cast<size_t>(E) * sizeof(uint32_t) + 256;
}

cudaError_t launch_permute(const int32_t* topk_idx, const void* x, int T, int H, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm, void* scratch,
                           uint32_t* err, cudaStream_t stream) {
  if (permute_is_small(T, E, k)) {
    long long g = static_cast<long long>(T) * k;  // one CTA per copied row, up to 4 per SM
    if (g > 4 * 148) g = 4 * 148;
    if (g < 1) g = 1;
    return launch_kernel(permute_small_kernel, dim3(static_cast<unsigned>(g)), dim3(kSmallThreads), 0, stream,
                         topk_idx, static_cast<const uint4*>(x), T, H / 8, E, k, counts, offsets, perm, inv,
                         static_cast<uint4*>(x_perm), err);
  }
  const int W = (T + 31) / 32;
  uint32_t* bitmap = static_cast<uint32_t*>(scratch);
  uint32_t* rowbase = bitmap + static_cast<size_t>(W) * E;
  const int threads = kWarpsPerBlock * 32;
  cudaError_t e = launch_kernel(bitmap_kernel, dim3((W + kWarpsPerBlock - 1) / kWarpsPerBlock), dim3(threads), 0,
                                stream, topk_idx, T, E, k, W, bitmap, err);
  if (e != cudaSuccess) return e;
  e = launch_kernel(scan_kernel, dim3(1), dim3(1024), 0, stream, bitmap, W, E, counts, offsets, rowbase);
  if (e != cudaSuccess) return e;
  const dim3 ggrid((T + kWarpsPerBlock - 1) / kWarpsPerBlock, (H / 8 + 31) / 32);
  return launch_kernel(gather_kernel, ggrid, dim3(threads), 0, stream, topk_idx, static_cast<const uint4*>(x), T,
                       H / 8, E, k, bitmap, rowbase, perm, inv, static_cast<uint4*>(x_perm), err);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// moe_permute_noalloc: the same three kernels with their scratch (the token
// bitmaps and row bases) in a fixed array that lives in this library's device
// image, so the caller passes no scratch and nothing is allocated.

namespace {

// Words per scratch array; the permute needs ceil(T/32) * E words for each of
// its two arrays, so calls with ceil(T/32) * E <= kNoAllocWords fit
// (for example T <= 8192 with E = 256, or T <= 262144 with E = 8).
constexpr size_t kNoAllocWords = 65536;

// 2 x 256 KiB, held by every GPU that loads the library until the process exits.
static __device__ __align__(256) uint32_t g_noalloc_scratch[2 * kNoAllocWords];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
moe_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" MOE_API moe_status_t moe_permute_noalloc(const int32_t* topk_idx, const void* x, int T, int H, int E,
                                                    int k, int32_t* counts, int32_t* offsets, int32_t* perm,
                                                    int32_t* inv, void* x_perm, moe_stream_t stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_VALUE;
  if (k > E || E > 256 || k > 16 || H % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  const size_t words = (static_cast<size_t>(T) + 31) / 32 * static_cast<size_t>(E);
  if (words > kNoAllocWords) return MOE_ERR_WORKSPACE;  // beyond the built-in scratch
  if (!counts || !offsets) return MOE_ERR_INVALID_VALUE;
  if (T > 0 && (!topk_idx || !x || !perm || !inv || !x_perm)) return MOE_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x_perm) & 15u))
    return MOE_ERR_INVALID_VALUE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  moe_status_t st = noalloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  // The device error word must exist before anything is launched: without it
  // an out-of-range expert id would be dropped silently.
  uint32_t* err = moe::device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  // Every scratch word the kernels read is written earlier in the same call
  // (bitmap_kernel writes all ceil(T/32) * E bitmap words, scan_kernel all
  // row bases), so nothing needs clearing between calls.
  const cudaError_t e = moe::launch_permute(topk_idx, x, T, H, E, k, counts, offsets, perm, inv, x_perm, scratch,
                                            err, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
