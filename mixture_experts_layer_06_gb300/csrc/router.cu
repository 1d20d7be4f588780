// Router scoring + top-k selection, one launch.
//
// "Cross-Platform Fused MoE Dispatch in Triton" (review page), "The reading":
// every token is first scored by the router; "Assumptions & free parameters":
// the standard softmax/sigmoid router with top-k selection.
//
// router_kernel: a cluster of C CTAs per tile of 128 tokens.  CTA r of the
// cluster computes the partial logits x . [W_r; w_s]^T over its share of the
// K = H columns on the 5th-generation tensor cores (tcgen05.mma, operands
// staged by TMA, fp32 accumulator in TMEM).  Large batches with a wide router
// run as C CTA pairs per tile of 256 tokens instead (cta_group::2: each CTA
// of a pair holds 128 token rows and half of the W_r rows, so every CTA
// streams half as many W_r bytes per token); everything below then happens
// within each half of the pairs.  CTA r owns tokens
// [r*128/C, (r+1)*128/C) of the tile: every CTA stores its partial logits of
// a token into the owner's shared memory (distributed shared memory stores,
// slot = source rank, column-major so that a warp's stores are contiguous),
// the owner adds the C partials in rank order, and a team of 8 lanes per
// owned token applies the logit bias and the score function, the optional
// group limit, and picks the k best experts (ties to the lower expert
// index).  Deterministic; no partial logits go to global memory.
// With a sigmoid-gated shared expert the gate vector w_s rides along as one
// more B row (its logit column gives the gate), else shared_gate_kernel.
#include <cfloat>
#include <climits>

#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

// warp 0: TMA, warp 1: MMA + TMEM owner; then every warp takes part in the
// TMEM -> shared memory exchange (warp w: TMEM lane quadrant w % 4, column
// part w / 4), the reduction and the selection (64 teams of 8 lanes: the 64
// tokens a CTA owns at a 2-way K split take one pass).
constexpr int kThreads = 512;
constexpr int kMaxStages = 8;
constexpr int kMaxCluster = 8;
constexpr int kPairMinT = 4096;  // batches from which the router runs as CTA pairs (router_plan)
constexpr int kTileM = 128;    // tokens per cluster
constexpr int kTileK = 64;     // bf16 elements per 128-byte swizzled row
constexpr int kATileBytes = kTileM * kTileK * 2;
constexpr int kBoxBytes = 16 * kTileK * 2;  // one 16-row box of B rows

struct RouterArgs {
  int T, H, E, k, NE, n_wr_boxes, gate_box, gate_col, stages, tmem_cols, kb_per_cta;
  RouteSpec spec;
  int32_t* topk_idx;
  float* topk_w;
  float* shared_scale;
  uint32_t* err;
};

// The partial-logit slots R[C][NE][ld] (column-major per source slot: the
// tokens of one logit column are contiguous, so a warp's stores of a column
// are one contiguous run) with ld = 128/C + 4: a multiple of 4 times an odd
// number modulo 32 banks, so that the 8-lane teams of the selection, reading
// experts tl, tl + 8, ... of 4 tokens, touch 32 distinct banks.  Then room for
// the logit bias of up to 256 experts.
__host__ __device__ constexpr int logit_ld(int C) { return kTileM / C + 4; }
__host__ __device__ constexpr int logit_buffer_bytes(int NE, int C) { return C * NE * logit_ld(C) * 4 + 256 * 4; }

constexpr int kTeam = 8;  // lanes that select the experts of one token

__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Team (8-lane butterfly) merges: the best two, or the best four in
// descending order, of the values the lanes hold.
__device__ __forceinline__ void team_top2(float& b1, float& b2) {
#pragma unroll
  for (int o = kTeam / 2; o > 0; o >>= 1) {
    const float p1 = __shfl_xor_sync(0xFFFFFFFFu, b1, o), p2 = __shfl_xor_sync(0xFFFFFFFFu, b2, o);
    b2 = fmaxf(fminf(b1, p1), fmaxf(b2, p2));
    b1 = fmaxf(b1, p1);
  }
}
__device__ __forceinline__ void team_top4(float (&c)[4]) {
  // the best four of two descending lists: bitonic half cleaner, then a
  // 4-element bitonic sort
#pragma unroll
  for (int o = kTeam / 2; o > 0; o >>= 1) {
    float d[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) d[j] = fmaxf(c[j], __shfl_xor_sync(0xFFFFFFFFu, c[3 - j], o));
    float x;
    x = fmaxf(d[0], d[2]); d[2] = fminf(d[0], d[2]); d[0] = x;
    x = fmaxf(d[1], d[3]); d[3] = fminf(d[1], d[3]); d[1] = x;
    x = fmaxf(d[0], d[1]); d[1] = fminf(d[0], d[1]); d[0] = x;
    x = fmaxf(d[2], d[3]); d[3] = fminf(d[2], d[3]); d[2] = x;
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = d[j];
  }
}
__device__ __forceinline__ void insert_top4(float (&c)[4], float v) {
  float m;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    m = fminf(c[j], v);
    c[j] = fmaxf(c[j], v);
    v = m;
  }
  c[3] = fmaxf(c[3], v);
}

// k rounds over a lane's NJ candidate logits lv[] (-inf = none; expert_of(j)
// = the expert of register j, increasing in j): each lane offers its best
// remaining candidate (a tree arg-max, adjacent pairs first so that among
// equal logits the lower register -- the lower expert -- wins), the team's
// best wins the round and its lane drops it.  The weights are the scores of
// the k winners (renormalised softmax: exp(v - v0), the denominator cancels);
// lane tl keeps rounds tl and tl + 8.
struct RoundsOut {
  float sum, s_lo, s_hi;
  int i_lo, i_hi;
};
template <int NJ, typename ExpertOf, typename Score>
__device__ __forceinline__ RoundsOut topk_rounds(float (&lv)[NJ], int k, int tl, bool renorm_softmax,
                                                 ExpertOf expert_of, Score score) {
  RoundsOut o{0.f, 0.f, 0.f, -1, -1};
  float v0 = 0.f;
  for (int r = 0; r < k; ++r) {
    float bv[NJ];
    int bj[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      bv[j] = lv[j];
      bj[j] = j;
    }
#pragma unroll
    for (int s = 1; s < NJ; s <<= 1)
#pragma unroll
      for (int l = 0; l + s < NJ; l += 2 * s) {
        const bool right = bv[l + s] > bv[l];
        bv[l] = right ? bv[l + s] : bv[l];
        bj[l] = right ? bj[l + s] : bj[l];
      }
    float v = bv[0];
    const int jb = bj[0];
    const bool has = v != -INFINITY;
    int i = has ? expert_of(jb) : INT_MAX;
    const int mine = i;
#pragma unroll
    for (int off = kTeam / 2; off > 0; off >>= 1) {
      const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, off);
      const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, off);
      if (better(v2, i2, v, i)) {
        v = v2;
        i = i2;
      }
    }
    if (has && i == mine) {
#pragma unroll
      for (int j = 0; j < NJ; ++j) lv[j] = j == jb ? -INFINITY : lv[j];
    }
    if (r == 0) v0 = v;
    const float sc = renorm_softmax ? __expf(v - v0) : score(v);
    o.sum += sc;
    if (r == tl) {
      o.s_lo = sc;
      o.i_lo = i;
    } else if (r == tl + kTeam) {
      o.s_hi = sc;
      o.i_hi = i;
    }
  }
  return o;
}

// The k best experts of one token by a team of 8 lanes (tl = lane within the
// team), from its summed logits L[e * ld] and the logit bias (both in shared
// memory; bias may be null).  Lane tl holds the logits of experts tl + 8j,
// j < JN (JN * 8 >= E), in registers, read once.  The score functions are
// monotone, so experts (and a group's top scores) are ranked by logit; scores
// are evaluated only where a value is needed.  Ties go to the lower expert
// (group) index.  M > 0: the groups are E / n_group = 8M experts wide, so
// group g is registers [gM, (g+1)M) of every lane and its best logits come
// from registers; M = 0: any group width, read from shared memory.  Every
// lane of the warp calls this (the shuffles span the warp); only `active`
// teams write.
template <int JN, int M>
__device__ void select_team(const float* L, int ld, const float* bias, const RouterArgs& a, int t, int tl,
                            bool active) {
  const int E = a.E, k = a.k;
  const bool sigmoid = a.spec.sigmoid != 0;
  auto logit = [&](int e) { return bias != nullptr ? L[e * ld] + bias[e] : L[e * ld]; };
  if (active && tl == 0 && a.gate_col >= 0) a.shared_scale[t] = 1.f / (1.f + __expf(-L[a.gate_col * ld]));
  const int ng = a.spec.n_group > 1 ? a.spec.n_group : 1;
  const int gsize = E / ng;

  float lv[JN];
#pragma unroll
  for (int j = 0; j < JN; ++j) {
    const int e = tl + kTeam * j;
    lv[j] = e < E ? logit(e) : -INFINITY;
  }

  // Softmax normaliser over all E logits, when a softmax score is used
  // un-renormalised or inside a group score.
  float mx = -INFINITY, inv_se = 1.f;
  if (!sigmoid && (!a.spec.renormalize || ng > 1)) {
#pragma unroll
    for (int j = 0; j < JN; ++j) mx = fmaxf(mx, lv[j]);
#pragma unroll
    for (int o = kTeam / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    float se = 0.f;
#pragma unroll
    for (int j = 0; j < JN; ++j) se += __expf(lv[j] - mx);  // exp(-inf) = 0 past E
#pragma unroll
    for (int o = kTeam / 2; o > 0; o >>= 1) se += __shfl_xor_sync(0xFFFFFFFFu, se, o);
    inv_se = 1.f / se;
  }
  auto score = [&](float v) { return sigmoid ? 1.f / (1.f + __expf(-v)) : __expf(v - mx) * inv_se; };

  // Group limit: group score = sum of the scores of its group_topn best
  // logits; the topk_group best groups are kept.  Lane tl holds the scores of
  // groups tl and tl + 8 (n_group <= 16).
  uint32_t kept = 0xFFFFFFFFu;
  if (ng > 1) {
    float gs_lo = -INFINITY, gs_hi = -INFINITY;
    const int n = a.spec.group_topn;
    if constexpr (M > 0) {
#pragma unroll
      for (int g = 0; g < JN / M; ++g) {
        if (g < ng) {
          float sg;
          if (n <= 2) {
            float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
            for (int q = 0; q < M; ++q) {
              const float v = lv[g * M + q];
              b2 = fmaxf(b2, fminf(b1, v));
              b1 = fmaxf(b1, v);
            }
            team_top2(b1, b2);
            sg = score(b1) + (n > 1 ? score(b2) : 0.f);
          } else {
            float c[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int q = 0; q < M; ++q) insert_top4(c, lv[g * M + q]);
            team_top4(c);
            sg = score(c[0]) + score(c[1]) + score(c[2]) + (n > 3 ? score(c[3]) : 0.f);
          }
          if (g == tl) gs_lo = sg;
          if (g == tl + kTeam) gs_hi = sg;
        }
      }
    } else {
      if (n <= 2) {
        // the group loop is unrolled so the merges of different groups
        // overlap their shuffle latencies
#pragma unroll 4
        for (int g = 0; g < ng; ++g) {
          float b1 = -INFINITY, b2 = -INFINITY;
          for (int e = g * gsize + tl; e < (g + 1) * gsize; e += kTeam) {
            const float v = logit(e);
            b2 = fmaxf(b2, fminf(b1, v));
            b1 = fmaxf(b1, v);
          }
          team_top2(b1, b2);
          const float sg = score(b1) + (n > 1 ? score(b2) : 0.f);
          if (g == tl) gs_lo = sg;
          if (g == tl + kTeam) gs_hi = sg;
        }
      } else {
        for (int g = 0; g < ng; ++g) {
          float c[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // this lane's best four, descending
          for (int e = g * gsize + tl; e < (g + 1) * gsize; e += kTeam) insert_top4(c, logit(e));
          team_top4(c);
          const float sg = score(c[0]) + score(c[1]) + score(c[2]) + (n > 3 ? score(c[3]) : 0.f);
          if (g == tl) gs_lo = sg;
          if (g == tl + kTeam) gs_hi = sg;
        }
      }
    }
    kept = 0;
    for (int r = 0; r < a.spec.topk_group; ++r) {
      // the best group not kept yet: this lane's candidate, then the team's
      const bool lo_ok = tl < ng && !((kept >> tl) & 1u), hi_ok = tl + kTeam < ng && !((kept >> (tl + kTeam)) & 1u);
      float v = lo_ok ? gs_lo : -INFINITY;
      int i = lo_ok ? tl : INT_MAX;
      if (hi_ok && (i == INT_MAX || gs_hi > v)) {
        v = gs_hi;
        i = tl + kTeam;
      }
#pragma unroll
      for (int o = kTeam / 2; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, o);
        if (better(v2, i2, v, i)) {
          v = v2;
          i = i2;
        }
      }
      if (i != INT_MAX) kept |= 1u << i;
    }
    // only the experts of kept groups stay candidates
    if constexpr (M > 0) {
#pragma unroll
      for (int j = 0; j < JN; ++j)
        if (!((kept >> (j / M)) & 1u)) lv[j] = -INFINITY;
    } else {
      int g = 0, gend = gsize;
#pragma unroll
      for (int j = 0; j < JN; ++j) {
        const int e = tl + kTeam * j;
        if (e < E) {
          while (e >= gend) {
            ++g;
            gend += gsize;
          }
          if (!((kept >> g) & 1u)) lv[j] = -INFINITY;
        }
      }
    }
  }

  const bool renorm_softmax = !sigmoid && a.spec.renormalize && ng == 1;
  RoundsOut o;
  if constexpr (M > 0) {
    if (ng > 1 && a.spec.topk_group * M <= JN / 2) {
      // The kept groups' candidates, compacted into half the registers (slot
      // s = the s-th kept group in ascending order, so register order still
      // follows expert order); the rounds then scan half as many values.
      constexpr int CJ = JN / 2, NS = CJ / M;
      float cv[CJ];
      unsigned long long gpack = 0;  // 4 bits per slot: its group (n_group <= 16)
      uint32_t rem = kept;
#pragma unroll
      for (int sl = 0; sl < NS; ++sl) {
        const int g = rem != 0 ? __ffs(rem) - 1 : -1;
        rem &= rem - 1;
        gpack |= static_cast<unsigned long long>(g & 15) << (4 * sl);
#pragma unroll
        for (int q = 0; q < M; ++q) {
          float v = -INFINITY;
#pragma unroll
          for (int g2 = 0; g2 < JN / M; ++g2) v = g == g2 ? lv[g2 * M + q] : v;
          cv[sl * M + q] = v;
        }
      }
      auto expert_of = [gpack, gsize, tl](int j) {
        const int g = static_cast<int>((gpack >> (4 * (j / M))) & 15u);
        return g * gsize + tl + kTeam * (j % M);
      };
      o = topk_rounds(cv, k, tl, renorm_softmax, expert_of, score);
    } else {
      o = topk_rounds(lv, k, tl, renorm_softmax, [tl](int j) { return tl + kTeam * j; }, score);
    }
  } else {
    o = topk_rounds(lv, k, tl, renorm_softmax, [tl](int j) { return tl + kTeam * j; }, score);
  }
  const float scale = a.spec.renormalize ? a.spec.route_scale / o.sum : a.spec.route_scale;
  if (active) {
    if (tl < k) {
      a.topk_idx[static_cast<size_t>(t) * k + tl] = o.i_lo;
      a.topk_w[static_cast<size_t>(t) * k + tl] = o.s_lo * scale;
    }
    if (tl + kTeam < k) {
      a.topk_idx[static_cast<size_t>(t) * k + tl + kTeam] = o.i_hi;
      a.topk_w[static_cast<size_t>(t) * k + tl + kTeam] = o.s_hi * scale;
    }
  }
}

// select_team with the register count JN for E and, where the groups line up
// with the lanes' strides, the register-resident group layout.
__device__ __forceinline__ void select_experts(const float* L, int ld, const float* bias, const RouterArgs& a, int t,
                                               int tl, bool active) {
  const int E = a.E;
  const int ng = a.spec.n_group > 1 ? a.spec.n_group : 1;
  const int m = (ng > 1 && (E / ng) % kTeam == 0) ? (E / ng) / kTeam : 0;
  if (E > 16 * kTeam) {
    if (m == 4)
      select_team<32, 4>(L, ld, bias, a, t, tl, active);
    else if (m == 2)
      select_team<32, 2>(L, ld, bias, a, t, tl, active);
    else if (m == 1)
      select_team<32, 1>(L, ld, bias, a, t, tl, active);
    else
      select_team<32, 0>(L, ld, bias, a, t, tl, active);
  } else if (E > 8 * kTeam) {
    select_team<16, 0>(L, ld, bias, a, t, tl, active);
  } else if (E > 4 * kTeam) {
    select_team<8, 0>(L, ld, bias, a, t, tl, active);
  } else if (E > 2 * kTeam) {
    select_team<4, 0>(L, ld, bias, a, t, tl, active);
  } else if (E > kTeam) {
    select_team<2, 0>(L, ld, bias, a, t, tl, active);
  } else {
    select_team<1, 0>(L, ld, bias, a, t, tl, active);
  }
}

// PAIR: the CTAs run as pairs (tcgen05 cta_group::2; one kernel may not mix
// the two CTA granularities).
template <bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_wr,
                  const __grid_constant__ CUtensorMap map_ws, const RouterArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  constexpr bool pair = PAIR;
  // B rows per CTA: all NE, or half of them on each CTA of a pair
  const int stage_bytes = kATileBytes + (pair ? a.NE / 2 : a.NE) * kTileK * 2;
  const uint32_t CL = gridDim.x;         // cluster size: the cluster spans blockIdx.x
  const uint32_t C = pair ? CL / 2 : CL;  // CTAs (pairs) splitting K
  const int region = max(S * stage_bytes, logit_buffer_bytes(a.NE, static_cast<int>(C)));
  float* P = reinterpret_cast<float*>(smem);  // summed / partial logits, after the last MMA
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + region);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0;
  const uint32_t kr = pair ? rank >> 1 : rank;  // K share
  const uint32_t phalf = pair ? rank & 1 : 0;   // a pair's CTA: token rows [128 phalf, +128) of the pair's 256
  const uint32_t even = rank & ~1u;             // the pair's even CTA (cluster rank)
  const int m0 = blockIdx.y * (pair ? 2 * kTileM : kTileM) + static_cast<int>(phalf) * kTileM;
  const int KB = a.H / kTileK;
  const int kb0 = static_cast<int>(kr) * a.kb_per_cta;
  const int kb1 = min(KB, kb0 + a.kb_per_cta);
  const int nboxes = a.n_wr_boxes + (a.gate_box >= 0 ? 1 : 0);

  pdl_trigger();
  // x belongs to earlier work of the stream; waiting before the TMEM
  // allocation also means a kernel never holds TMEM while an earlier one on
  // the same SM may still need some.
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
    if (pair) {
      tmem_alloc_pair(tmem_holder, a.tmem_cols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_holder, a.tmem_cols);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (pair) cluster_sync();  // the pair's barriers exist before any remote use
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    // Lane 0: wait for the slot, post the bytes, load the x tile, the W_r rows
    // (one box) and, with a fused gate, the w_s row (one 16-row box).
    // A pair: each CTA loads its 128 token rows and its half of the W_r rows
    // (map_wr's box is NE/2 rows), both completing on the even CTA's barrier.
    if (lane == 0) {
      int issued = 0;
      int s = 0;         // ring slot and phase of stage `issued` (running counters)
      uint32_t ph = 0;
      for (int kb = kb0; kb < kb1; ++kb, ++issued) {
        if (!mbar_wait(&empty[s], ph ^ 1, a.err, kSiteRouterProducer)) break;
        uint8_t* st = smem + s * stage_bytes;
        if (pair) {
          if (phalf == 0) mbar_arrive_expect_tx(&full[s], 2u * static_cast<uint32_t>(stage_bytes));
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), even);
          tma_load_2d_pair(st, &map_x, bar, kb * kTileK, m0);
          tma_load_2d_pair(st + kATileBytes, &map_wr, bar, kb * kTileK, static_cast<int>(phalf) * (a.NE / 2));
        } else {
          mbar_arrive_expect_tx(&full[s], kATileBytes + nboxes * kBoxBytes);
          tma_load_2d(st, &map_x, &full[s], kb * kTileK, m0);
          tma_load_2d(st + kATileBytes, &map_wr, &full[s], kb * kTileK, 0);
          if (a.gate_box >= 0)
            tma_load_2d(st + kATileBytes + a.gate_box * kBoxBytes, &map_ws, &full[s], kb * kTileK, 0);
        }
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
      // Do not leave while copies into this CTA's shared memory are in flight
      // (a pair's loads complete on the even CTA: wait until they were consumed).
      for (int i = (issued > S ? issued - S : 0); i < issued; ++i) {
        if (pair)
          mbar_wait(&empty[i % S], (i / S) & 1, a.err, kSiteTeardown);
        else
          mbar_wait(&full[i % S], (i / S) & 1, a.err, kSiteTeardown);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && phalf == 0) {  // a pair's MMAs are issued by its even CTA
      const uint32_t idesc = idesc_bf16_f32(pair ? 2 * kTileM : kTileM, a.NE);
      int s = 0;
      uint32_t ph = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[s], ph, a.err, kSiteRouterMma)) break;
        tc_fence_after_sync();
        const uint32_t a_addr = smem_u32(smem + s * stage_bytes);
        const uint32_t b_addr = a_addr + kATileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileK / 16; ++kk) {
          if (pair)
            umma_bf16_pair(tmem_base, sdesc_k128(a_addr + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                           (kb != kb0 || kk != 0));
          else
            umma_bf16(tmem_base, sdesc_k128(a_addr + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                      (kb != kb0 || kk != 0));
        }
        if (pair)
          umma_commit_pair_at(&empty[s], even);
        else
          umma_commit(&empty[s]);
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
      if (pair)
        umma_commit_pair_at(acc_full, even);
      else
        umma_commit(acc_full);
    }
    __syncwarp();
  }
  // Every CTA of the cluster reaches every cluster barrier, whatever happened
  // above (a wait that gave up has recorded the error and the role stopped).
  // Barrier 1: every MMA of the cluster has completed (every warp waited for
  // its own accumulator), so every CTA's pipeline stages are free to receive
  // partial logits.
  bool acc_ok = mbar_wait(acc_full, 0, a.err, kSiteRouterEpilogue);
  acc_ok = __all_sync(0xFFFFFFFFu, acc_ok);  // the TMEM loads below are warp-collective
  tc_fence_after_sync();
  __syncthreads();
  if (CL > 1) cluster_sync();

  // Thread = token row (TMEM lane): its NE partial logits go to the CTA that
  // owns the row, into slot `kr` of that CTA's buffer R[C][NE][ld] (with
  // pairs: the CTA of the same pair half in the owning pair).
  const int rpc = kTileM / static_cast<int>(C);
  const int ld = logit_ld(static_cast<int>(C));
  const int slot_floats = a.NE * ld;
  // Column parts: NE split into 4 (NE a multiple of 128), 2 (of 64) or 1;
  // warp w takes part w / 4 of its lane quadrant's columns.
  const int parts = a.NE % 128 == 0 ? 4 : a.NE % 64 == 0 ? 2 : 1;
  const int part = warp >> 2;
  if (acc_ok && part < parts) {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int cbeg = part * (a.NE / parts), cend = cbeg + a.NE / parts;
    const uint32_t owner = static_cast<uint32_t>(row / rpc);  // its K share index
    const int rr = row - static_cast<int>(owner) * rpc;  // row within the owner's share
    float* slot = P + static_cast<size_t>(kr) * slot_floats;
    const uint32_t dst = smem_u32(slot + rr);
    const bool local = owner == kr || C == 1;
    const uint32_t dst_c = local ? dst : mapa_shared(dst, pair ? 2 * owner + phalf : owner);
    for (int c0 = cbeg; c0 < cend; c0 += 32) {
      uint32_t r[32];
      const uint32_t ta = tmem_addr(tmem_base, q * 32, c0);
      if (cend - c0 >= 32)
        tmem_ld32(ta, r);
      else
        tmem_ld16(ta, r);
      tmem_wait(r);
      const int nc = min(32, cend - c0);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nc) {
          if (local)
            slot[(c0 + i) * ld + rr] = __uint_as_float(r[i]);
          else
            asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst_c + 4u * (c0 + i) * ld), "r"(r[i])
                         : "memory");
        }
    }
  }
  tc_fence_before_sync();
  // Barrier 2: every partial row has arrived.  After it no CTA touches
  // another's shared memory.
  __syncthreads();
  if (CL > 1) cluster_sync();

  // Owned rows: add the C partials in rank order into slot 0.
  if (C > 1) {
    // 4 consecutive rows of one column per thread (rpc and ld are multiples of 4)
    const int q4 = rpc / 4, n = q4 * a.NE;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const int c = i / q4, r = (i - c * q4) * 4;
      float4* dst = reinterpret_cast<float4*>(P + c * ld + r);
      float4 v = *dst;
      for (int src = 1; src < static_cast<int>(C); ++src) {
        const float4 w = *reinterpret_cast<const float4*>(P + src * slot_floats + c * ld + r);
        v.x += w.x;
        v.y += w.y;
        v.z += w.z;
        v.w += w.w;
      }
      *dst = v;
    }
    __syncthreads();
  }
  // The logit bias, staged once per CTA after the partial-logit slots (when given).
  float* bias_s = nullptr;
  if (a.spec.logit_bias != nullptr) {
    bias_s = P + static_cast<int>(C) * slot_floats;
    for (int e = threadIdx.x; e < a.E; e += kThreads) bias_s[e] = a.spec.logit_bias[e];
    __syncthreads();
  }
  // Selection: team i of 8 lanes takes owned rows i, i + kTeams, ...
  constexpr int kTeams = kThreads / kTeam;
  const int team = threadIdx.x / kTeam, tl = threadIdx.x % kTeam;
  for (int base = 0; base < rpc; base += kTeams) {
    if (base + (threadIdx.x & ~31) / kTeam >= rpc) break;  // whole warp past the owned rows
    const int r = base + team, t = m0 + static_cast<int>(kr) * rpc + r;
    const bool active = r < rpc && t < a.T;
    const float* L = P + (r < rpc ? r : 0);
    select_experts(L, ld, bias_s, a, t, tl, active);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    if (pair)
      tmem_dealloc_pair(tmem_base, a.tmem_cols);
    else
      tmem_dealloc(tmem_base, a.tmem_cols);
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

// Decode-sized batches (T <= kTinyT, router weights of at most kTinyWr
// elements, x of at most kTinyX): routing and the grouping onto experts in
// one CTA, one launch.
//  1. the T rows of x into shared memory; logits[t][e] = x[t] . W_r[e] (and
//     x[t] . w_s for a gated shared expert): one warp per column, each
//     weight row read once, on the CUDA cores, fp32 accumulation of the
//     bf16 products, 16-byte loads;
//  2. score, group limit and top-k by the same 8-lane team routine as
//     router_kernel;
//  3. counts, offsets (exclusive scan) and, for copy q = t*k + j of expert e,
//     its grouped row offsets[e] + #{earlier tokens that chose e} (stable);
//  4. perm, inv, and the x rows copied to x_perm.
constexpr int kTinyT = 8;
constexpr int kTinyWr = 128 * 1024;  // E * H
constexpr int kTinyX = 48 * 1024;    // T * H: the batch's x rows, staged in shared memory (96 KB at most)
constexpr int kTinyThreads = 512;

struct TinyArgs {
  RouterArgs r;
  const __nv_bfloat16* x;
  const __nv_bfloat16* w_router;
  const __nv_bfloat16* w_shared_gate;
  int32_t *counts, *offsets, *perm, *inv;
  uint4* x_perm;
};

// fp32 sum of the products of 8 bf16 pairs (one 16-byte load of each), into acc.
__device__ __forceinline__ void fma8_bf16(const uint4& xa, const uint4& wa, float& acc) {
  const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xa);
  const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wa);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 xf = __bfloat1622float2(xp[i]), wf = __bfloat1622float2(wp[i]);
    acc = fmaf(xf.x, wf.x, acc);
    acc = fmaf(xf.y, wf.y, acc);
  }
}

// out[t] = xs[t] . w for the T token rows in shared memory (xs: T rows of
// H/8 16-byte vectors), by one warp (H a multiple of 8), fp32.  The weight row
// is read once, in chunks of 8 vectors per lane held in registers while a
// runtime loop over the tokens adds each token's partial dot product (warp
// reduction, lane 0 accumulates into out).  The code stays short: this
// one-CTA kernel runs once per forward from a cold instruction cache, and
// fully unrolled variants measured slower (Mixtral-shaped T=1, logits of 8
// experts: 12 / 19 / 32 us with 4 / 8 / 16 loads in flight when the loop was
// also unrolled over every token, 5 us with one load at a time).
__device__ __noinline__ void column_tiny(const uint4* xs, const __nv_bfloat16* w, int T, int H, int lane,
                                         float* out) {
  constexpr int kU = 8;
  const uint4* wv = reinterpret_cast<const uint4*>(w);
  const int n = H / 8;
  if (lane < T) out[lane] = 0.f;
  __syncwarp();
  for (int c0 = 0; c0 < n; c0 += 32 * kU) {
    const int v0 = c0 + lane;
    uint4 wa[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (v0 + 32 * u < n) wa[u] = wv[v0 + 32 * u];
    for (int t = 0; t < T; ++t) {
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (v0 + 32 * u < n) fma8_bf16(xs[t * n + v0 + 32 * u], wa[u], acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (lane == 0) out[t] += acc;
    }
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kTinyThreads, 1) route_permute_tiny_kernel(const TinyArgs ta) {
  __shared__ float logits[(256 + 16) * kTinyT];  // column-major: logits[e * kTinyT + t]
  __shared__ float bias_s[256];
  __shared__ int32_t idx_s[kTinyT * 16];
  __shared__ int32_t off_s[257];
  __shared__ int32_t row_s[kTinyT * 16];  // grouped row of copy q
  extern __shared__ uint4 x_s[];          // the batch's x rows, T x H/8 vectors
  pdl_trigger();
  pdl_wait();
  const RouterArgs& a = ta.r;
  const int T = a.T, E = a.E, k = a.k, H = a.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncol = E + (ta.w_shared_gate != nullptr ? 1 : 0);  // the gate is column E
  const int H8 = H / 8;
  {
    // x into shared memory, four loads in flight per thread
    const uint4* xg = reinterpret_cast<const uint4*>(ta.x);
    const int total = T * H8;
    for (int i0 = threadIdx.x; i0 < total; i0 += 4 * kTinyThreads) {
      uint4 val[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * kTinyThreads < total) val[u] = xg[i0 + u * kTinyThreads];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u * kTinyThreads < total) x_s[i0 + u * kTinyThreads] = val[u];
    }
  }
  __syncthreads();
  // One warp per column, against every token's x from shared memory.
  for (int e = warp; e < ncol; e += kTinyThreads / 32) {
    const __nv_bfloat16* w = e < E ? ta.w_router + static_cast<size_t>(e) * H : ta.w_shared_gate;
    column_tiny(x_s, w, T, H, lane, logits + e * kTinyT);
  }
  if (a.spec.logit_bias != nullptr)
    for (int e = threadIdx.x; e < E; e += kTinyThreads) bias_s[e] = a.spec.logit_bias[e];
  __syncthreads();
  // selection: team i of 8 lanes takes token i (the routine's gate column is column E)
  {
    const int team = threadIdx.x / kTeam, tl = threadIdx.x % kTeam;
    if (warp < (T + 3) / 4) {  // warps holding at least one token's team
      const bool active = team < T;
      select_experts(logits + (active ? team : 0), kTinyT, a.spec.logit_bias != nullptr ? bias_s : nullptr, a,
                     team, tl, active);
    }
  }
  __syncthreads();  // topk_idx written to global memory by the teams
  for (int q = threadIdx.x; q < T * k; q += kTinyThreads) idx_s[q] = a.topk_idx[q];
  __syncthreads();
  // counts and offsets (E <= 256: thread e counts; a serial scan by thread 0)
  if (threadIdx.x < E) {
    int c = 0;
    for (int q = 0; q < T * k; ++q) c += idx_s[q] == static_cast<int>(threadIdx.x);
    off_s[threadIdx.x] = c;
    ta.counts[threadIdx.x] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      const int c = off_s[e];
      off_s[e] = run;
      run += c;
    }
    off_s[E] = run;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += kTinyThreads) ta.offsets[e] = off_s[e];
  // grouped row of copy q: stable in token order
  auto row_of = [&](int q) {
    const int t = q / k, e = idx_s[q];
    int r = off_s[e];
    for (int q2 = 0; q2 < t * k; ++q2) r += idx_s[q2] == e;
    return r;
  };
  for (int q = threadIdx.x; q < T * k; q += kTinyThreads) {
    const int r = row_of(q);
    ta.perm[r] = q;
    ta.inv[q] = r;
    row_s[q] = r;
  }
  __syncthreads();
  // x_perm: the T*k copies of the staged rows
  const int total = T * k * H8;
  for (int i = threadIdx.x; i < total; i += kTinyThreads) {
    const int q = i / H8, v = i - q * H8;
    ta.x_perm[static_cast<size_t>(row_s[q]) * H8 + v] = x_s[(q / k) * H8 + v];
  }
}

}  // namespace

RouterPlan router_plan(int T, int H, int E, bool shared_gate) {
  RouterPlan p{};
  const int ne_wr = (E + 15) / 16 * 16;
  p.fused_gate = shared_gate && ne_wr + 16 <= 256;
  p.NE = ne_wr + (p.fused_gate ? 16 : 0);
  // CTA pairs for large batches with a wide router: every 128-token tile
  // re-reads all of W_r from L2, and a pair (M = 256 tokens per MMA) halves
  // that; each CTA of a pair holds half of the NE rows of B, so the fused
  // shared-expert gate row, which must sit with the W_r rows, is not paired.
  p.pair = !p.fused_gate && p.NE >= 128 && T >= kPairMinT;
  const int rows = p.pair ? 2 * kTileM : kTileM;
  p.m_tiles = (T + rows - 1) / rows;
  const int KB = H / kTileK;
  // The largest power-of-two K split c (a cluster of c CTAs, or c pairs;
  // at most 8 CTAs) that keeps the grid within one wave of ~152 CTAs and
  // leaves every CTA at least two K blocks, so that the W_r stream of a small
  // batch spreads over several SMs.  Unpaired, clusters of 8 only while the
  // grid stays within half the SMs: measured on GB300, the DeepSeek-V3-shaped router at
  // T=2048 (16 token tiles) takes 58 us in clusters of 8 (128 CTAs) and
  // 38 us in clusters of 4, while at T=512 (4 tiles, 32 CTAs) 8 beats 4
  // (34 vs 38 us), as it does for every smaller router measured (Mixtral-,
  // Qwen2- and skew-shaped layers, T=32..512).  Shapes only.
  const int per = p.pair ? 2 : 1;
  int c = 1;
  while (per * c < kMaxCluster && p.m_tiles * per * (2 * c) <= 152 && KB / (2 * c) >= 2 &&
         !(per == 1 && 2 * c >= kMaxCluster && p.m_tiles * (2 * c) > 76))
    c <<= 1;
  p.kb_per_cta = (KB + c - 1) / c;
  while (c > 1 && (c - 1) * p.kb_per_cta >= KB) c >>= 1;  // every CTA gets a K block
  p.kb_per_cta = (KB + c - 1) / c;
  p.ksplit = c;
  p.cluster = per * c;
  return p;
}

bool route_permute_is_tiny(int T, int H, int E, int k) {
  return T >= 1 && T <= kTinyT && static_cast<long long>(E) * H <= kTinyWr && T * H <= kTinyX && E <= 256 &&
         k <= 16;
}

cudaError_t launch_route_permute_tiny(int T, int H, int E, int k, const RouteSpec& spec, const void* x,
                                      const void* w_router, const void* w_shared_gate, int32_t* topk_idx,
                                      float* topk_w, float* shared_scale, int32_t* counts, int32_t* offsets,
                                      int32_t* perm, int32_t* inv, void* x_perm, cudaStream_t stream) {
  TinyArgs t{};
  t.r.T = T;
  t.r.H = H;
  t.r.E = E;
  t.r.k = k;
  const bool gate = w_shared_gate != nullptr && shared_scale != nullptr;
  t.r.gate_col = gate ? E : -1;
  t.r.spec = spec;
  t.r.topk_idx = topk_idx;
  t.r.topk_w = topk_w;
  t.r.shared_scale = shared_scale;
  t.x = static_cast<const __nv_bfloat16*>(x);
  t.w_router = static_cast<const __nv_bfloat16*>(w_router);
  t.w_shared_gate = gate ? static_cast<const __nv_bfloat16*>(w_shared_gate) : nullptr;
  t.counts = counts;
  t.offsets = offsets;
  t.perm = perm;
  t.inv = inv;
  t.x_perm = static_cast<uint4*>(x_perm);
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(route_permute_tiny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTinyX * 2);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const size_t smem = static_cast<size_t>(T) * H * 2;  // the staged x rows
  return launch_kernel(route_permute_tiny_kernel, dim3(1), dim3(kTinyThreads), smem, stream, t);
}

int router_launches(int T, int H, int E, bool shared_gate) {
  if (T == 0) return 0;
  const RouterPlan p = router_plan(T, H, E, shared_gate);
  return 1 + ((shared_gate && !p.fused_gate) ? 1 : 0);
}

cudaError_t launch_router(const CUtensorMap& map_x, const CUtensorMap& map_wr, const CUtensorMap* map_ws, int T,
                          int H, int E, int k, const RouteSpec& spec, const void* x, const void* w_shared_gate,
                          int32_t* topk_idx, float* topk_w, float* shared_scale, uint32_t* err,
                          cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const bool gate = w_shared_gate != nullptr && shared_scale != nullptr;
  const RouterPlan p = router_plan(T, H, E, gate);
  RouterArgs g{};
  g.T = T;
  g.H = H;
  g.E = E;
  g.k = k;
  g.NE = p.NE;
  g.n_wr_boxes = (E + 15) / 16;
  g.gate_box = p.fused_gate ? g.n_wr_boxes : -1;
  g.gate_col = p.fused_gate ? g.n_wr_boxes * 16 : -1;
  g.tmem_cols = p.NE <= 32 ? 32 : p.NE <= 64 ? 64 : p.NE <= 128 ? 128 : 256;
  g.kb_per_cta = p.kb_per_cta;
  g.spec = spec;
  g.topk_idx = topk_idx;
  g.topk_w = topk_w;
  g.shared_scale = shared_scale;
  g.err = err;
  const int stage_bytes = kATileBytes + (p.pair ? p.NE / 2 : p.NE) * kTileK * 2;
  const int fixed = 1024 + (2 * kMaxStages + 2) * 8 + 64;
  int stages = (227 * 1024 - fixed) / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages > p.kb_per_cta) stages = p.kb_per_cta;
  g.stages = stages;
  const int lbuf = logit_buffer_bytes(p.NE, p.ksplit);
  const int region = stages * stage_bytes > lbuf ? stages * stage_bytes : lbuf;
  // At least half an SM's shared memory, so that one router CTA at most runs
  // on an SM: a CTA that waits at a cluster barrier then never holds TMEM
  // another cluster's CTA on the same SM is waiting to allocate.
  size_t smem = static_cast<size_t>(fixed) + static_cast<size_t>(region);
  if (smem < 116 * 1024) smem = 116 * 1024;

  static bool configured[2][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kernel = p.pair ? router_kernel<true> : router_kernel<false>;
  if (dev < 64 && !configured[p.pair][dev]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured[p.pair][dev] = true;
  }
  const dim3 grid(p.cluster, p.m_tiles);
  cudaError_t e = launch_kernel_cluster(kernel, grid, dim3(kThreads), smem, stream, p.cluster, map_x, map_wr,
                                        p.fused_gate ? *map_ws : map_wr, g);
  if (e != cudaSuccess) return e;
  if (gate && !p.fused_gate) {
    e = launch_kernel(shared_gate_kernel, dim3((T * 32 + 255) / 256), dim3(256), 0, stream,
                      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_shared_gate), T, H,
                      shared_scale);
  }
  return e;
}

}  // namespace moe
