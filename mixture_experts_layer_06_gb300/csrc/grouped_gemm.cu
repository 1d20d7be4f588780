// Persistent grouped GEMM for the expert FFN on the 5th-generation tensor cores.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "What carries
// the argument": the gate and up projections of a SwiGLU expert are computed
// from one shared load of each input tile and SiLU(gate)*up is finished in
// registers, so the two intermediates never reach global memory; the rest is
// a grouped GEMM over (expert, token-offset) blocks.  The page's design maps a
// fixed block size onto a schedule built on the host; here the schedule is
// built on the device, inside every CTA, from the scanned expert offsets, and
// the CTAs are persistent, so skewed routing spreads a hot expert's tiles over
// all SMs instead of stranding them ("Load-bearing premise" / the Zipf skew
// study name that failure mode).
//
// Orientation: weights are the MMA's A operand (M = 128 weight rows of one
// expert), tokens are B (N = bn tokens, 16..256), so a tile with few tokens
// still runs a full-height MMA and streams weights at full width.  D^T tiles
// live in TMEM: lane = weight row, column = token.
//   SwiGLU (or GEGLU: GELU in place of SiLU, chosen per segment):
//            the 128-row A tile stacks 64 gate rows over the 64 up rows of
//            the same features (one TMA box over a view in which gate and up
//            are two planes), so ONE accumulator of bn columns holds both
//            projections of a tile and two accumulator slots fit in TMEM:
//            the epilogue of one tile overlaps the MMAs of the next.  The
//            epilogue warps that read the gate lanes and the up lanes of the
//            same features trade half of each 32-column chunk through shared
//            memory and each finishes h = SiLU(g) * u for its half -> bf16.
//   Store:   128 output rows per CTA -> fp16 (the down projection's expert
//            outputs, K-split slices at small batches), fp32, or bf16 (the
//            unfused gate / up projections of the fusion ablation).
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-5 epilogue (warp w reads TMEM lanes 32*(w%4)..+31).
// Pipelines: a ring of `stages` shared-memory slots (full/empty mbarriers) and
// two TMEM accumulator slots (tmem_full/tmem_empty mbarriers).  Every wait is
// bounded; a wait that gives up records a device error and its role stops.
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

// Exact MMA width (compile-time): a token tile with fewer than bn rows runs
// its MMAs with N = its rows rounded up to 16 (else N = bn).
#ifndef MOE_EXACT_N
#define MOE_EXACT_N 1
#endif

// L2 cache policies on the TMA loads: token rows evict-last, a weight tile
// read by a single token tile evict-first, other weight tiles normal (0: all
// normal).
#ifndef MOE_L2_HINTS
#define MOE_L2_HINTS 1
#endif


constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kTileM = 128;
constexpr int kTileK = 64;
constexpr int kATileBytes = kTileM * kTileK * 2;  // 16 KB
constexpr int kMaxSegGroups = 256;
constexpr int kHalfRows = 64;                    // SwiGLU: gate rows (= up rows) per A tile
constexpr int kHalfBytes = kHalfRows * kTileK * 2;  // 8 KB
// Epilogue shared memory.  Store: per-warp 32x32 fp32 transpose tiles.
// SwiGLU: the exchange slots [warp pair][slot][half][lane][16 fp32] and
// per-warp 16x32 bf16 output tiles.
constexpr int kStoreStagingBytes = 4 * 32 * 32 * 4;
constexpr int kXchgBytes = 2 * 2 * 2 * 32 * 16 * 4;
constexpr int kSwiGLUStagingBytes = kXchgBytes + 4 * 16 * 32 * 2;
__host__ __device__ constexpr int staging_bytes(int epi) {
  return epi == kEpiSwiGLU ? kSwiGLUStagingBytes : kStoreStagingBytes;
}
// Output rows (features) per CTA and tile: 64 for SwiGLU (the A tile holds
// their gate and up rows), 128 for the plain store.
__host__ __device__ constexpr int feat_per_cta(int epi) { return epi == kEpiSwiGLU ? kHalfRows : kTileM; }

struct SegDev {
  const int32_t* offsets;
  int groups, rows, nout, K, bn, ldo, ksplit;
  int a_mode;    // SwiGLU A loads: kStackedMap or kTwoMaps
  int up_first;  // stacked map: plane 0 is the up weights (lanes 0-63 = up)
  int gelu;      // gated epilogue: GELU (erf form) instead of SiLU
  size_t slice_stride;
  void* out;
  int kstages;   // stages of kps K blocks in the full K
};

struct GemmArgs {
  SegDev seg[2];
  int nseg;
  int munit;  // output features per tile: NSUB * feat_per_cta(epi), x2 for a CTA pair
  int stages;
  int kps;  // 64-wide K blocks per pipeline stage (one 3-D TMA box each)
  int bn_max;
  int acc_cols;  // TMEM columns per accumulator slot: NSUB * bn_max
  int nslots;    // accumulator slots (2: the epilogue of a tile overlaps the next tile's MMAs)
  int mix;       // spread segment 1's tiles evenly between segment 0's (see decode_tile)
  int tmem_cols;
  uint32_t* err;
};

struct Sched {
  int prefix[2][kMaxSegGroups + 1];    // first tile of each group
  int rowstart[2][kMaxSegGroups + 1];  // first B row of each group; [G] = end
  int trows[2][kMaxSegGroups];         // token rows per tile of each group | token tiles << 10
  int seg_end[2];                      // tile count after segment 0 / 1
};

// SiLU(g) = g / (1 + exp(-g)) with the fast divide; the input is clamped so
// that the divisor stays finite (SiLU(-80) is 0 to far below bf16 resolution).
__device__ __forceinline__ float silu(float g) {
  return __fdividef(g, 1.f + __expf(-fmaxf(g, -80.f)));
}

// GELU(g) = g/2 * (1 + erf(g / sqrt(2))), the exact form (GEGLU experts).
__device__ __forceinline__ float gelu_erf(float g) { return 0.5f * g * (1.f + erff(g * 0.70710678118654752f)); }

// h = act(g) * u for the 16 columns a warp finishes, into its bf16 staging
// tile: own[j] are this warp's values, peer[j] its partner's.
template <bool GELU>
__device__ __forceinline__ void gated16(const uint32_t (&v)[32], const float (&peer)[16], int half, bool own_gate,
                                        __nv_bfloat16* st, int lane) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float own = __uint_as_float(half ? v[16 + j] : v[j]);
    const float gv = own_gate ? own : peer[j], uv = own_gate ? peer[j] : own;
    st[j * 32 + lane] = __float2bfloat16_rn((GELU ? gelu_erf(gv) : silu(gv)) * uv);
  }
}

struct GemmMaps {
  SegMaps seg[2];
};

// Index of the token box a tile loads: the smallest of the segment's boxes
// (bstep, 2 bstep, ...) that covers the tile's rows per CTA.  The producer
// and the MMA issuer must agree on it: with several K blocks per stage, the
// blocks of one box lie box-rows * 128 bytes apart in shared memory.
#ifndef MOE_EXACT_BOX
#define MOE_EXACT_BOX 1
#endif
__device__ __forceinline__ int box_index(const SegMaps& ms, int rows_per_cta) {
  if (!MOE_EXACT_BOX) return ms.nb - 1;
  return min(max((rows_per_cta + ms.bstep - 1) / ms.bstep - 1, 0), ms.nb - 1);
}

struct Tile {
  int s, g, mb, tb, a_row, b_row, valid, bn, kb0, kb1;
  int ntb;  // token tiles of the group (each streams the same weight tiles)
  size_t out_off;  // element offset of this tile's output slice
};

// With two segments, position p of the tile sequence is a segment-1 tile
// when floor((p + 1) n1 / n) > floor(p n1 / n) (n tiles, n1 of segment 1):
// the shared expert's tiles (few weight bytes, all compute) are spread
// evenly between the routed experts' tiles (weight streaming) instead of
// running after them, so the weight stream and the tensor work overlap over
// the whole launch.  Only when segment 1's token rows are small next to L2
// (launch_grouped_gemm): measured on GB300, interleaving the Qwen2-shaped
// shared expert (T=512, 3.7 MB of token rows) took its gate+up GEMM from 495
// to 447 us, but interleaving the DeepSeek-V3-shaped one at T=8192 (117 MB
// of token rows, re-read by every feature block) slowed it from 3600 to
// 3790 us: its rows no longer stay in L2 between uses.
#ifndef MOE_MIX_SEGMENTS
#define MOE_MIX_SEGMENTS 1
#endif
// A role's place in its walk over the tiles: the group of the last tile it
// decoded in each segment.  A role visits its tiles in increasing order, and
// so (also with segments mixed) increasing within each segment, so the group
// of the next tile is found by scanning forward from there.
struct WalkHint {
  int g0, g1;  // segment 0, segment 1 (two scalars: an indexed pair would live in local memory)
};

__device__ __forceinline__ Tile decode_tile(const GemmArgs& a, const Sched& sc, int tile, WalkHint& h) {
  Tile t;
  if (MOE_MIX_SEGMENTS && a.nseg > 1 && a.mix) {
    const long long n = sc.seg_end[1], n1 = n - sc.seg_end[0];
    const int c0 = static_cast<int>(static_cast<long long>(tile) * n1 / n);
    const int c1 = static_cast<int>(static_cast<long long>(tile + 1) * n1 / n);
    tile = c1 > c0 ? sc.seg_end[0] + c0 : tile - c0;
  }
  t.s = (a.nseg > 1 && tile >= sc.seg_end[0]) ? 1 : 0;
  const SegDev& sg = a.seg[t.s];
  const int* pre = sc.prefix[t.s];
  int g = t.s ? h.g1 : h.g0;  // the last group with pre[g] <= tile (empty groups are passed over)
  while (g + 1 < sg.groups && pre[g + 1] <= tile) ++g;
  if (t.s)
    h.g1 = g;
  else
    h.g0 = g;
  t.g = g;
  int local = tile - pre[g];
  const int rows_g = sc.rowstart[t.s][g + 1] - sc.rowstart[t.s][g];
  t.bn = sg.bn;
  int ks = 0;  // K slice, fastest
  if (sg.ksplit > 1) {
    ks = local % sg.ksplit;
    local /= sg.ksplit;
  }
  const int packed = sc.trows[t.s][g];
  const int tr = packed & 1023, ntb = packed >> 10;
  t.ntb = ntb;
  if (ntb == 1) {
    t.mb = local;
    t.tb = 0;
  } else {
    t.mb = local / ntb;
    t.tb = local - t.mb * ntb;
  }
  t.a_row = g * sg.nout + t.mb * a.munit;
  t.b_row = sc.rowstart[t.s][g] + t.tb * tr;
  t.valid = min(tr, rows_g - t.tb * tr);
  const int KB = sg.kstages;
  if (sg.ksplit > 1) {
    t.kb0 = ks * KB / sg.ksplit;
    t.kb1 = (ks + 1) * KB / sg.ksplit;
  } else {
    t.kb0 = 0;
    t.kb1 = KB;
  }
  t.out_off = static_cast<size_t>(ks) * sg.slice_stride;
  return t;
}

// Tile schedule from the group offsets; run by one warp.
__device__ void build_schedule(const GemmArgs& a, Sched& sc) {
  const int lane = threadIdx.x & 31;
  int total = 0;
  for (int s = 0; s < a.nseg; ++s) {
    const SegDev& sg = a.seg[s];
    const int mblocks = sg.nout / a.munit;
    for (int base = 0; base < sg.groups; base += 32) {
      const int g = base + lane;
      int start = 0, rows_g = 0;
      if (g < sg.groups) {
        if (sg.offsets != nullptr) {
          start = sg.offsets[g];
          rows_g = sg.offsets[g + 1] - start;
        } else {
          rows_g = sg.rows;
        }
        // Clamp corrupt offsets so that no tile reaches outside the segment.
        start = min(max(start, 0), sg.rows);
        rows_g = min(max(rows_g, 0), sg.rows - start);
      }
      // The token tiles of a group are balanced (equal rows, rounded up to
      // 16), so that the tiles sharing a weight block stream it through L2
      // in step instead of a short last tile racing ahead.
      const int ntb = (rows_g + sg.bn - 1) / sg.bn;
      const int tiles = (g < sg.groups) ? mblocks * ntb * sg.ksplit : 0;
      if (g < sg.groups)
        sc.trows[s][g] = (ntb > 0 ? ((rows_g + ntb - 1) / ntb + 15) / 16 * 16 : sg.bn) | (max(ntb, 1) << 10);
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      if (g < sg.groups) {
        sc.prefix[s][g] = total + incl - tiles;
        sc.rowstart[s][g] = start;
        if (g == sg.groups - 1) sc.rowstart[s][g + 1] = start + rows_g;
      }
      total += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) {
      sc.prefix[s][sg.groups] = total;
      sc.seg_end[s] = total;
    }
  }
  if (lane == 0 && a.nseg == 1) sc.seg_end[1] = total;
}

// The kernel body.  PAIR: the two CTAs of a cluster work as one CTA pair
// (tcgen05 cta_group::2): a tile covers 2 x feat_per_cta(EPI) output features,
// CTA r holds the A rows of its half of them and token rows
// [N/2 r, N/2 r + N/2) of B, the even CTA issues the M=256 MMAs for both and
// every TMA load of the pair completes on the even CTA's full barrier.  Each
// CTA receives its 128 rows of D in its own TMEM and runs its own epilogue.
template <int EPI, bool PAIR, int NSUB>
__device__ __forceinline__ void gemm_body(const GemmMaps& maps, const GemmArgs& a) {
  constexpr bool SWIGLU = (EPI == kEpiSwiGLU);
  constexpr int BDIV = PAIR ? 2 : 1;  // share of the token rows held by one CTA
  constexpr int FEAT = feat_per_cta(EPI);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const int KPS = a.kps;
  const int stage_bytes = KPS * (NSUB * kATileBytes + (a.bn_max / BDIV) * kTileK * 2);
  uint8_t* staging = smem + S * stage_bytes;
  Sched* sched = reinterpret_cast<Sched*>(staging + staging_bytes(EPI));
  uint64_t* full = reinterpret_cast<uint64_t*>(sched + 1);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* xfull = tempty + 2;  // SwiGLU: [warp pair][slot], both warps' values written
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(xfull + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;
  const int first = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int stride = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  pdl_trigger();
  if (threadIdx.x == 64) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4 * BDIV);  // every epilogue warp of the pair
    }
    for (int i = 0; i < 4; ++i) mbar_init(&xfull[i], 64);
    fence_mbar_init();
  }
  // The offsets, the token rows and the outputs belong to earlier work of the
  // stream.  Waiting before the TMEM allocation also means a kernel never
  // holds TMEM while an earlier one on the same SM may still need some.
  pdl_wait();
  if (warp == 1) {
    __syncwarp();
    if (PAIR) {
      tmem_alloc_pair(tmem_holder, a.tmem_cols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, a.tmem_cols);
      tmem_relinquish();
    }
  }
  if (warp == 0) build_schedule(a, *sched);
  tc_fence_before_sync();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers exist before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const Sched& sc = *sched;
  const int total = sc.seg_end[a.nseg - 1];

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // One elected lane: wait for a free slot, post the byte count, issue the
    // loads of the weight tile and of the token tile.  The token rows come in
    // one request per stage through the smallest of the segment's box heights
    // that covers this CTA's share of the tile (box_index); rows past the
    // tile's own are not used.  Several smaller boxes per tile were measured
    // to be much slower.
    int it = 0;
    if (lane == 0) {
      for (int sg = 0; sg < a.nseg; ++sg) {
        tma_prefetch_map(&maps.seg[sg].a0);
        if (SWIGLU && a.seg[sg].a_mode == kTwoMaps) tma_prefetch_map(&maps.seg[sg].a1);
        for (int i = 0; i < maps.seg[sg].nb; ++i) tma_prefetch_map(&maps.seg[sg].b[i]);
      }
      // L2 policies: token rows are re-read by every weight block of their
      // group (evict last); a weight tile read by one token tile only is
      // streamed (evict first), one shared by several stays normal.
      const uint64_t p_first = MOE_L2_HINTS ? l2_policy_evict_first() : l2_policy_evict_normal();
      const uint64_t p_normal = l2_policy_evict_normal();
      const uint64_t pb = MOE_L2_HINTS ? l2_policy_evict_last() : l2_policy_evict_normal();
      bool ok = true;
      int ps = 0;        // ring slot of stage `it` (it % S, kept as a running counter:
      uint32_t pph = 0;  // a division per stage is not free on the issue path) and its phase
      WalkHint hint{0, 0};
      for (int tile = first; tile < total && ok; tile += stride) {
        const Tile t = decode_tile(a, sc, tile, hint);
        const SegMaps& ms = maps.seg[t.s];
        const bool two_maps = SWIGLU && a.seg[t.s].a_mode == kTwoMaps;  // then KPS == 1
        const int n_tile = MOE_EXACT_N ? ((t.valid + 15) >> 4) << 4 : t.bn;
        const int a_row = t.a_row + static_cast<int>(rank) * FEAT * NSUB;
        const int b_row = t.b_row + static_cast<int>(rank) * (n_tile / BDIV);
        // the smallest token box that covers this CTA's n_tile / BDIV rows
        const int bi = box_index(ms, n_tile / BDIV);
        const CUtensorMap* mb = &ms.b[bi];
        const uint64_t pa = t.ntb == 1 ? p_first : p_normal;
        const uint32_t bytes = BDIV * KPS * (NSUB * kATileBytes + (bi + 1) * ms.bstep * kTileK * 2);
        for (int kb = t.kb0; kb < t.kb1; ++kb, ++it) {
          const int s = ps;
          const uint32_t ph = pph;
          if (++ps == S) {
            ps = 0;
            pph ^= 1;
          }
          if (!mbar_wait(&empty[s], ph ^ 1, a.err, kSiteGemmProducer)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * stage_bytes;
          uint8_t* sb = st + KPS * NSUB * kATileBytes;
          if (PAIR) {
            if (rank == 0) mbar_arrive_expect_tx(&full[s], bytes);
            const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
            if (two_maps) {
              for (int u = 0; u < NSUB; ++u) {
                tma_load_2d_pair_hint(st + u * kATileBytes, &ms.a0, bar, kb * kTileK, a_row + u * kHalfRows, pa);
                tma_load_2d_pair_hint(st + u * kATileBytes + kHalfBytes, &ms.a1, bar, kb * kTileK,
                                      a_row + u * kHalfRows, pa);
              }
            } else if (SWIGLU) {
              for (int u = 0; u < NSUB; ++u) {  // sub-tile u: its KPS A tiles, KPS * 16 KB
                uint8_t* dst = st + u * KPS * kATileBytes;
                if (KPS == 1)
                  tma_load_3d_pair_hint(dst, &ms.a0, bar, kb * kTileK, a_row + u * kHalfRows, 0, pa);
                else
                  tma_load_4d_pair_hint(dst, &ms.a0, bar, 0, a_row + u * kHalfRows, 0, kb * KPS, pa);
              }
            } else {
              for (int u = 0; u < NSUB; ++u) {  // sub-tile u: 128 weight rows, KPS * 16 KB
                uint8_t* dst = st + u * KPS * kATileBytes;
                if (KPS == 1)
                  tma_load_2d_pair_hint(dst, &ms.a0, bar, kb * kTileK, a_row + u * kTileM, pa);
                else
                  tma_load_3d_pair_hint(dst, &ms.a0, bar, 0, a_row + u * kTileM, kb * KPS, pa);
              }
            }
            if (KPS == 1)
              tma_load_2d_pair_hint(sb, mb, bar, kb * kTileK, b_row, pb);
            else
              tma_load_3d_pair_hint(sb, mb, bar, 0, b_row, kb * KPS, pb);
          } else {
            mbar_arrive_expect_tx(&full[s], bytes);
            if (two_maps) {
              for (int u = 0; u < NSUB; ++u) {
                tma_load_2d_hint(st + u * kATileBytes, &ms.a0, &full[s], kb * kTileK, a_row + u * kHalfRows, pa);
                tma_load_2d_hint(st + u * kATileBytes + kHalfBytes, &ms.a1, &full[s], kb * kTileK,
                                 a_row + u * kHalfRows, pa);
              }
            } else if (SWIGLU) {
              for (int u = 0; u < NSUB; ++u) {
                uint8_t* dst = st + u * KPS * kATileBytes;
                if (KPS == 1)
                  tma_load_3d_hint(dst, &ms.a0, &full[s], kb * kTileK, a_row + u * kHalfRows, 0, pa);
                else
                  tma_load_4d_hint(dst, &ms.a0, &full[s], 0, a_row + u * kHalfRows, 0, kb * KPS, pa);
              }
            } else {
              for (int u = 0; u < NSUB; ++u) {
                uint8_t* dst = st + u * KPS * kATileBytes;
                if (KPS == 1)
                  tma_load_2d_hint(dst, &ms.a0, &full[s], kb * kTileK, a_row + u * kTileM, pa);
                else
                  tma_load_3d_hint(dst, &ms.a0, &full[s], 0, a_row + u * kTileM, kb * KPS, pa);
              }
            }
            if (KPS == 1)
              tma_load_2d_hint(sb, mb, &full[s], kb * kTileK, b_row, pb);
            else
              tma_load_3d_hint(sb, mb, &full[s], 0, b_row, kb * KPS, pb);
          }
        }
      }
      // Do not leave while copies into this CTA's shared memory are in flight:
      // wait until the last stages were consumed (their loads had landed).
      for (int i = (it > S ? it - S : 0); i < it; ++i) {
        if (PAIR)
          mbar_wait(&empty[i % S], (i / S) & 1, a.err, kSiteTeardown);
        else
          mbar_wait(&full[i % S], (i / S) & 1, a.err, kSiteTeardown);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {
      int n = 0;
      int ms_ = 0;       // ring slot and phase of the next stage (running counters)
      uint32_t mph = 0;
      bool ok = true;
      WalkHint hint{0, 0};
      for (int tile = first; tile < total && ok; tile += stride, ++n) {
        const Tile t = decode_tile(a, sc, tile, hint);
        const int acc = a.nslots == 2 ? (n & 1) : 0;
        const uint32_t aph = (a.nslots == 2 ? (n >> 1) : n) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1, a.err, kSiteGemmMma)) break;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + acc * a.acc_cols;
        const int n_tile = MOE_EXACT_N ? ((t.valid + 15) >> 4) << 4 : t.bn;
        const uint32_t idesc = idesc_bf16_f32(kTileM * BDIV, n_tile);
        // consecutive K blocks of the token box lie box-rows * 128 bytes apart
        const SegMaps& ms = maps.seg[t.s];
        const uint32_t b_atom = (box_index(ms, n_tile / BDIV) + 1) * ms.bstep * kTileK * 2;
        for (int kb = t.kb0; kb < t.kb1; ++kb) {
          const int s = ms_;
          const uint32_t ph = mph;
          if (++ms_ == S) {
            ms_ = 0;
            mph ^= 1;
          }
          if (!mbar_wait(&full[s], ph, a.err, kSiteGemmMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = smem_u32(smem + s * stage_bytes);
          const uint32_t bb = a0 + KPS * NSUB * kATileBytes;
          for (int j = 0; j < KPS; ++j) {
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              const uint64_t bdesc = sdesc_k128(bb + j * b_atom + kk * 32);
              const uint32_t accum = (kb != t.kb0 || j != 0 || kk != 0);
              for (int u = 0; u < NSUB; ++u) {  // sub-tile u: A tile u*KPS+j, accumulator at column u*bn_max
                const uint64_t adesc = sdesc_k128(a0 + (u * KPS + j) * kATileBytes + kk * 32);
                if (PAIR)
                  umma_bf16_pair(d + u * a.bn_max, adesc, bdesc, idesc, accum);
                else
                  umma_bf16(d + u * a.bn_max, adesc, bdesc, idesc, accum);
              }
            }
          }
          if (PAIR)
            umma_commit_pair(&empty[s]);
          else
            umma_commit(&empty[s]);
        }
        if (PAIR)
          umma_commit_pair(&tfull[acc]);
        else
          umma_commit(&tfull[acc]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const uint32_t tempty_leader = PAIR ? mapa_shared(smem_u32(&tempty[0]), 0) : 0;
    // SwiGLU: warps q and q^2 read the gate and the up lanes of the same 32
    // features (lanes 32q.. and 32(q^2)..); the low-lane warp finishes token
    // columns [0,16) of every 32-column chunk, the other [16,32).
    const int half = q >> 1, pq = q & 1;
    float* xb = reinterpret_cast<float*>(staging) + pq * (2 * 2 * 32 * 16);
    uint8_t* stg = SWIGLU ? staging + kXchgBytes + (warp - 2) * (16 * 32 * 2) : staging + (warp - 2) * (32 * 32 * 4);
    uint32_t xseq = 0;  // exchange chunk counter (the same sequence in both warps of a pair)
    bool ok = true;
    int n = 0;
    WalkHint hint{0, 0};
    for (int tile = first; tile < total && ok; tile += stride, ++n) {
      const Tile t = decode_tile(a, sc, tile, hint);
      const int acc = a.nslots == 2 ? (n & 1) : 0;
      const uint32_t aph = (a.nslots == 2 ? (n >> 1) : n) & 1;
      if (!mbar_wait(&tfull[acc], aph, a.err, kSiteGemmEpilogue)) break;
      tc_fence_after_sync();
      const SegDev& sg = a.seg[t.s];
      const uint32_t col0 = acc * a.acc_cols;
      const int ncols = MOE_EXACT_N ? ((t.valid + 15) >> 4) << 4 : t.bn;  // the columns the MMA wrote
      if constexpr (SWIGLU) {
        const bool own_gate = (half == 0) != (sg.up_first != 0);
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.out);
        __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stg);
        // sub-tile u: features u*64.., accumulator at column u*bn_max
        for (int u = 0; u < NSUB && ok; ++u) {
          for (int c0 = 0; c0 < ncols; c0 += 32, ++xseq) {
            const int feat0 = t.mb * a.munit + static_cast<int>(rank) * FEAT * NSUB + u * FEAT + pq * 32;
            const int nc = min(32, ncols - c0);
            uint32_t v[32];
            const uint32_t ta = tmem_addr(tmem_base, q * 32, col0 + u * a.bn_max + c0);
            if (nc == 32)
              tmem_ld32(ta, v);
            else
              tmem_ld16(ta, v);
            tmem_wait(v);
            const int slot = xseq & 1;
            float* send = xb + (slot * 2 + half) * (32 * 16) + lane * 16;
            const float* recv = xb + (slot * 2 + (half ^ 1)) * (32 * 16) + lane * 16;
            const int sw = (lane >> 1) & 3;  // 16-byte swizzle: conflict-free rows of 64 bytes
            // Send the partner's 16 columns (none when the chunk has only 16 and
            // this is the low-lane warp).
            if (half == 1 || nc == 32) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                // constant register indices on both sides of the select
                const uint4 lo = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                const uint4 hi = make_uint4(v[16 + 4 * c], v[17 + 4 * c], v[18 + 4 * c], v[19 + 4 * c]);
                *reinterpret_cast<uint4*>(send + 4 * (c ^ sw)) = half ? lo : hi;
              }
            }
            mbar_arrive(&xfull[pq * 2 + slot]);
            if (!mbar_wait(&xfull[pq * 2 + slot], (xseq >> 1) & 1, a.err, kSiteGemmEpilogue)) {
              ok = false;
              break;
            }
            const int my0 = half * 16;
            if (my0 < nc) {
              float p[16];
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const float4 f = *reinterpret_cast<const float4*>(recv + 4 * (c ^ sw));
                p[4 * c] = f.x;
                p[4 * c + 1] = f.y;
                p[4 * c + 2] = f.z;
                p[4 * c + 3] = f.w;
              }
              if (sg.gelu)
                gated16<true>(v, p, half, own_gate, st, lane);
              else
                gated16<false>(v, p, half, own_gate, st, lane);
              __syncwarp();
              for (int w = lane; w < 16 * 4; w += 32) {
                const int j = w >> 2, piece = w & 3;
                const int r = c0 + my0 + j;
                const int row = t.b_row + r;
                if (r < t.valid && row < sg.rows)
                  *reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * sg.ldo + feat0 + piece * 8) =
                      *reinterpret_cast<const uint4*>(st + j * 32 + piece * 8);
              }
              __syncwarp();
            }
          }
        }
      } else if constexpr (EPI == kEpiStoreBF16 || EPI == kEpiStoreF16) {
        constexpr bool F16 = (EPI == kEpiStoreF16);
        uint16_t* out = static_cast<uint16_t*>(sg.out) + t.out_off;
        uint16_t* st = reinterpret_cast<uint16_t*>(stg);
        float amax = 0.f;
        for (int u = 0; u < NSUB; ++u) {
          const int feat0 = t.mb * a.munit + static_cast<int>(rank) * FEAT * NSUB + u * FEAT + q * 32;
          for (int c0 = 0; c0 < ncols; c0 += 32) {
            const int nc = min(32, ncols - c0);
            uint32_t g[32];
            const uint32_t ta = tmem_addr(tmem_base, q * 32, col0 + u * a.bn_max + c0);
            if (nc == 32)
              tmem_ld32(ta, g);
            else
              tmem_ld16(ta, g);
            tmem_wait(g);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nc) {
                const float v = __uint_as_float(g[j]);
                if constexpr (F16) {
                  amax = fmaxf(amax, fabsf(v));
                  st[j * 32 + lane] = __half_as_ushort(__float2half_rn(v));
                } else {
                  st[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                }
              }
            __syncwarp();
            for (int w = lane; w < nc * 4; w += 32) {
              const int j = w >> 2, piece = w & 3;
              const int row = t.b_row + c0 + j;
              if (c0 + j < t.valid && row < sg.rows)
                *reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * sg.ldo + feat0 + piece * 8) =
                    *reinterpret_cast<const uint4*>(st + j * 32 + piece * 8);
            }
            __syncwarp();
          }
        }
        // fp16 holds |v| <= 65504; anything larger (or NaN) is reported.
        if (F16 && !(amax <= 65504.f)) raise_error(a.err, kErrBounds, kSiteOverflow);
      } else {
        float* out = static_cast<float*>(sg.out) + t.out_off;
        float* st = reinterpret_cast<float*>(stg);
        // sub-tile u: weight rows u*128.., accumulator at column u*bn_max
        for (int u = 0; u < NSUB; ++u) {
          const int feat0 = t.mb * a.munit + static_cast<int>(rank) * FEAT * NSUB + u * FEAT + q * 32;
          for (int c0 = 0; c0 < ncols; c0 += 32) {
            const int nc = min(32, ncols - c0);
            uint32_t g[32];
            const uint32_t ta = tmem_addr(tmem_base, q * 32, col0 + u * a.bn_max + c0);
            if (nc == 32)
              tmem_ld32(ta, g);
            else
              tmem_ld16(ta, g);
            tmem_wait(g);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nc) st[j * 32 + lane] = __uint_as_float(g[j]);
            __syncwarp();
            for (int w = lane; w < nc * 8; w += 32) {
              const int j = w >> 3, piece = w & 7;
              const int row = t.b_row + c0 + j;
              if (c0 + j < t.valid && row < sg.rows)
                *reinterpret_cast<float4*>(out + static_cast<size_t>(row) * sg.ldo + feat0 + piece * 4) =
                    *reinterpret_cast<const float4*>(st + j * 32 + piece * 4);
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(tempty_leader + acc * 8);
        else
          mbar_arrive(&tempty[acc]);
      }
    }
  }

  __syncthreads();
  if (PAIR) cluster_sync();  // the pair is done with TMEM and with each other's barriers
  if (warp == 1) {
    tc_fence_after_sync();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, a.tmem_cols);
    else
      tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

// NSUB: sub-tiles per CTA and tile (SwiGLU: stacked 64-feature tiles; store: 128-row tiles).
template <int EPI, int NSUB>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmMaps maps,
                                                                    const GemmArgs a) {
  gemm_body<EPI, false, NSUB>(maps, a);
}

template <int EPI, int NSUB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
  gemm_body<EPI, true, NSUB>(maps, a);
}

template <typename K>
cudaError_t allow_big_smem(K kernel, bool* configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || configured[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e == cudaSuccess) configured[dev] = true;
  return e;
}

template <int EPI, int NSUB>
cudaError_t launch_epi(const GemmArgs& a, const GemmMaps& maps, int grid, size_t smem, bool pair,
                       cudaStream_t stream) {
  static bool single_ok[64] = {}, pair_ok[64] = {};
  cudaError_t e;
  if (pair) {
    if ((e = allow_big_smem(grouped_gemm_pair_kernel<EPI, NSUB>, pair_ok)) != cudaSuccess) return e;
    return launch_kernel(grouped_gemm_pair_kernel<EPI, NSUB>, dim3(grid), dim3(kThreads), smem, stream, maps, a);
  }
  if ((e = allow_big_smem(grouped_gemm_kernel<EPI, NSUB>, single_ok)) != cudaSuccess) return e;
  return launch_kernel(grouped_gemm_kernel<EPI, NSUB>, dim3(grid), dim3(kThreads), smem, stream, maps, a);
}

uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// Shared memory besides the pipeline stages: alignment slack, epilogue
// staging, the schedule, the barriers and the TMEM address.
constexpr int fixed_smem(int epi) {
  return 1024 + staging_bytes(epi) + static_cast<int>(sizeof(Sched)) + (2 * kMaxStages + 4 + 4) * 8 + 64;
}

// Epilogues whose partial sums may be cut into K slices.
constexpr bool k_splittable(int epi) { return epi == kEpiStoreF32 || epi == kEpiStoreF16; }

int bn_max_of(int num_segments, const GemmSegment* segs) {
  int m = 16;
  for (int s = 0; s < num_segments; ++s) m = m > segs[s].bn ? m : segs[s].bn;
  return m;
}

}  // namespace

// CTA pairs (tcgen05 cta_group::2) halve the token rows each CTA stages and
// reads, which is what limits the large-tile, tensor-bound GEMMs.  Measured on
// GB300: with 256-row token tiles the down projection runs 18-20 % faster as
// pairs (Mixtral T=4096, DeepSeek-V3 T=8192); with 128-row or smaller tiles
// pairs gain nothing or lose a little.
#ifndef MOE_PAIR_MIN_BN
#define MOE_PAIR_MIN_BN 256
#endif
// The same threshold for the SwiGLU GEMM, whose CTA holds 64 features: as a
// pair, a token tile is read once per 128 features instead of once per 64.
#ifndef MOE_PAIR_MIN_BN_SWIGLU
#define MOE_PAIR_MIN_BN_SWIGLU 256
#endif
// Largest number of 64-wide K blocks per pipeline stage (one 3-D / 4-D TMA
// box each); taken when at least MOE_MIN_STAGES stages still fit.
#ifndef MOE_KPS_MAX
#define MOE_KPS_MAX 2
#endif
#ifndef MOE_MIN_STAGES
#define MOE_MIN_STAGES 3
#endif
// Sub-tiles per CTA and tile (NSUB).  Small token tiles stream weights: two
// sub-tiles put more weight bytes per token byte into every stage (more
// weight bytes in flight per SM), and 2 x NSUB accumulators of bn columns
// must fit in TMEM's 512 columns, so 256-row tiles take one.  Measured on
// GB300: two sub-tiles gain 6-14 % on the SwiGLU GEMM at 128-row tiles and
// 8-11 % on the down projection at 64-128-row tiles (Mixtral-, Qwen2-,
// DeepSeek-V3-shaped layers).  But halving the tile count can leave a last
// wave of tiles on few SMs (Mixtral T=1: 224 tiles on 152 SMs), so two
// sub-tiles are taken only while the expected tiles still fill their waves.
#ifndef MOE_NSUB_SMALL
#define MOE_NSUB_SMALL 2  // token tiles of 16..128 rows
#endif
// 256-row token tiles: sub-tiles per CTA.  Two fill TMEM with one tile's
// accumulators (one slot: the epilogue no longer overlaps the next tile).
#ifndef MOE_NSUB_LARGE
#define MOE_NSUB_LARGE 1
#endif
#ifndef MOE_MIN_WAVE_FILL
#define MOE_MIN_WAVE_FILL 0.9
#endif

namespace {

// Sub-tiles the plan starts from for token tiles of bn_max rows.
int gemm_nsub(int bn_max) {
  int n = bn_max >= 256 ? MOE_NSUB_LARGE : MOE_NSUB_SMALL;
  while (n > 1 && n * bn_max > 512) n >>= 1;
  return n;
}

// Expected tiles of a launch (host estimate from the shapes: rows spread
// evenly over min(groups, rows) groups) and the fill of its last wave.
double wave_fill(GemmEpilogue epi, int num_segments, const GemmSegment* segs, int munit, int units) {
  long long tiles = 0;
  for (int s = 0; s < num_segments; ++s) {
    const GemmSegment& g = segs[s];
    const long long active = g.offsets == nullptr ? 1 : (g.rows < g.groups ? g.rows : g.groups);
    if (active <= 0) continue;
    const long long per = (g.rows + active - 1) / active;
    const int ks = (!k_splittable(epi) || g.ksplit < 1) ? 1 : g.ksplit;
    tiles += active * ((per + g.bn - 1) / g.bn) * (g.nout / munit) * ks;
  }
  if (tiles <= 0 || units <= 0) return 1.0;
  const long long waves = (tiles + units - 1) / units;
  return static_cast<double>(tiles) / static_cast<double>(waves * units);
}

}  // namespace

GemmPlan grouped_gemm_plan(GemmEpilogue epi, int num_segments, const GemmSegment* segs, int num_sms,
                           bool static_grid) {
  GemmPlan p{};
  const int bn_max = bn_max_of(num_segments, segs);
  const int feat = feat_per_cta(epi);
  p.nsub = static_grid ? 1 : gemm_nsub(bn_max);
  for (int s = 0; s < num_segments; ++s)
    while (p.nsub > 1 && segs[s].nout % (p.nsub * feat) != 0) p.nsub >>= 1;
  const int pair_min = epi == kEpiSwiGLU ? MOE_PAIR_MIN_BN_SWIGLU : MOE_PAIR_MIN_BN;
  p.pair = !static_grid && pair_min > 0 && bn_max >= pair_min;
  for (int s = 0; s < num_segments; ++s) p.pair = p.pair && segs[s].nout % (2 * p.nsub * feat) == 0;
  if (p.nsub > 1 && !p.pair) {
    const double fill = wave_fill(epi, num_segments, segs, feat * p.nsub, num_sms);
    if (fill < MOE_MIN_WAVE_FILL && wave_fill(epi, num_segments, segs, feat, num_sms) > fill) p.nsub = 1;
  }
  const int per_kb = p.nsub * kATileBytes + (p.pair ? bn_max / 2 : bn_max) * kTileK * 2;
  // Several sub-tiles: two-block stages pay even with two stages once the
  // token tiles reach 64 rows (measured on Mixtral-, Qwen2- and
  // DeepSeek-V3-shaped layers).
  const int min_stages = (p.nsub >= 2 && bn_max >= 64) ? 2 : MOE_MIN_STAGES;
  p.kps = 1;
  for (int cand = 2; cand <= MOE_KPS_MAX; cand <<= 1) {
    bool ok = (227 * 1024 - fixed_smem(epi)) / (cand * per_kb) >= min_stages;
    for (int s = 0; s < num_segments && ok; ++s) {
      const int ks = (!k_splittable(epi) || segs[s].ksplit < 1) ? 1 : segs[s].ksplit;
      ok = segs[s].K % (kTileK * cand) == 0 && segs[s].K / (kTileK * cand) >= 2 * ks;
      if (epi == kEpiSwiGLU && segs[s].a_mode == kTwoMaps) ok = false;  // two 2-D boxes per stage
    }
    if (ok) p.kps = cand;
  }
  return p;
}

cudaError_t launch_grouped_gemm(GemmEpilogue epi, int num_segments, const GemmSegment* segs, const SegMaps* seg_maps,
                                int num_sms, uint32_t* err, cudaStream_t stream, long long static_ctas) {
  const GemmPlan plan = grouped_gemm_plan(epi, num_segments, segs, num_sms, static_ctas > 0);
  GemmArgs a{};
  a.nseg = num_segments;
  a.err = err;
  a.munit = feat_per_cta(epi) * plan.nsub * (plan.pair ? 2 : 1);
  long long upper = 0;
  for (int s = 0; s < num_segments; ++s) {
    const GemmSegment& g = segs[s];
    const int ks = (!k_splittable(epi) || g.ksplit < 1) ? 1 : g.ksplit;
    a.seg[s] = SegDev{g.offsets, g.groups, g.rows, g.nout, g.K, g.bn, g.ldo, ks, g.a_mode, g.up_first, g.gelu,
                      g.slice_stride, g.out, g.K / (kTileK * plan.kps)};
    a.bn_max = a.bn_max > g.bn ? a.bn_max : g.bn;
    upper += static_cast<long long>(g.nout / a.munit) * ((g.rows + g.bn - 1) / g.bn + g.groups) * ks;
  }
  a.acc_cols = plan.nsub * a.bn_max;
  a.nslots = 2 * a.acc_cols <= 512 ? 2 : 1;
  a.mix = num_segments > 1 && static_cast<long long>(segs[1].rows) * segs[1].K * 2 <= (32ll << 20);
  a.tmem_cols = static_cast<int>(pow2_at_least(static_cast<uint32_t>(a.nslots * a.acc_cols)));
  a.kps = plan.kps;
  const int stage_bytes =
      a.kps * (plan.nsub * kATileBytes + (plan.pair ? a.bn_max / 2 : a.bn_max) * kTileK * 2);
  int stages = (227 * 1024 - fixed_smem(epi)) / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  a.stages = stages;
  const size_t smem = static_cast<size_t>(fixed_smem(epi)) + static_cast<size_t>(stages) * stage_bytes;
  int units = plan.pair ? num_sms / 2 : num_sms;  // CTAs, or CTA pairs
  if (upper < units) units = static_cast<int>(upper);
  if (static_ctas > 0) units = static_cast<int>(static_ctas < (1ll << 30) ? static_ctas : (1ll << 30));
  if (units < 1) units = 1;
  const int grid = plan.pair ? 2 * units : units;
  GemmMaps maps;
  maps.seg[0] = seg_maps[0];
  maps.seg[1] = seg_maps[num_segments > 1 ? 1 : 0];
  if (epi == kEpiSwiGLU) {
    if (plan.nsub == 2) return launch_epi<kEpiSwiGLU, 2>(a, maps, grid, smem, plan.pair, stream);
    return launch_epi<kEpiSwiGLU, 1>(a, maps, grid, smem, plan.pair, stream);
  }
  if (epi == kEpiStoreBF16) {
    if (plan.nsub == 2) return launch_epi<kEpiStoreBF16, 2>(a, maps, grid, smem, plan.pair, stream);
    return launch_epi<kEpiStoreBF16, 1>(a, maps, grid, smem, plan.pair, stream);
  }
  if (epi == kEpiStoreF16) {
    if (plan.nsub == 2) return launch_epi<kEpiStoreF16, 2>(a, maps, grid, smem, plan.pair, stream);
    return launch_epi<kEpiStoreF16, 1>(a, maps, grid, smem, plan.pair, stream);
  }
  if (plan.nsub == 2) return launch_epi<kEpiStoreF32, 2>(a, maps, grid, smem, plan.pair, stream);
  return launch_epi<kEpiStoreF32, 1>(a, maps, grid, smem, plan.pair, stream);
}

}  // namespace moe
