// K1: the single streaming pass over the verify logits (argmax for greedy
// verification, mini-sglang PR #134 verify.py; log-sum-exp for p(t) and q(t),
// spec-decode README "How it works").
//
// Persistent and warp-specialized. The rows of both logit sets form one
// flattened element space of T = rows * V elements; CTA g owns the elements
// [T g / G, T (g+1) / G), so every CTA streams the same number of bytes
// whatever the row count. Warp 0 is the producer: one lane walks the CTA's
// row pieces and issues 1-D bulk copies (TMA) of up to 16 KB into a 6-stage
// shared-memory ring, arming each stage's "full" mbarrier with the byte count
// and reusing a stage once all consumer warps have released it on its
// "empty" mbarrier. Warps 1..8 consume: each thread folds its group of 16-byte
// vectors of each stage into a running (max, sum 2^((x - max) c)) and
// remembers the group holding its first maximum. At the end of every row
// piece the consumers resolve the exact argmax, reduce (shuffles, then a
// named barrier across the consumer warps) and write one Partial per
// (CTA, row piece); the decide kernel merges a row's partials.
//
// Copies cover the 16-byte-aligned hull of each row piece when it lies inside
// the logit buffer, and elements outside the piece are masked in the first
// and last stage; only a piece touching an unaligned buffer start or end
// falls back to scalar loads for its ragged edge.
//
// Every wait is bounded (mbar_wait_bounded); a warp that gives up stops
// waiting, its CTA's remaining partials carry err = 1, and the producer waits
// (bounded) for its copies in flight before the CTA exits.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kK1Consumers = 8;                       // consumer warps
constexpr int kK1Threads = 32 * (kK1Consumers + 1);   // + one producer warp
constexpr int kK1ConsumerThreads = 32 * kK1Consumers;
constexpr int kK1StageBytes = 16384;
constexpr int kK1Stages = 6;
constexpr int kK1SmemBytes = kK1StageBytes * kK1Stages;
constexpr int kK1CtasPerSm = 2;
constexpr int kK1MaxCtas = 4096;                      // bound used to size the workspace
constexpr int kK1MinBytesPerCta = 16384;
// Vectors one consumer thread folds per stage.
constexpr int kGroupVecs = kK1StageBytes / 16 / kK1ConsumerThreads;
static_assert(kGroupVecs == 4, "fold_group assumes four vectors per thread and stage");

struct RowSet {
  const uint8_t* base;   // first row
  int64_t stride_bytes;  // row pitch
  int32_t rows;
  uintptr_t safe_lo;     // [safe_lo, safe_hi): bytes the caller's buffer holds
  uintptr_t safe_hi;
};

struct RowStatsArgs {
  RowSet set0;         // target rows
  RowSet set1;         // draft rows (rows = 0 if none)
  int32_t V;
  int64_t T;           // (set0.rows + set1.rows) * V
  int32_t G;           // CTAs
  float c;             // log2(e) / T
  Partial* partials;   // [rows + G]: slot row + cta, one per (CTA, row piece)
};

// CTA that owns flattened element e under the equal split of T elements:
// the largest g with floor(T g / G) <= e, i.e. with T g < (e + 1) G. A float
// estimate is corrected with exact 64-bit products (no 64-bit division).
__host__ __device__ __forceinline__ int cta_of(int64_t e, int64_t T, int G) {
  int g = static_cast<int>(static_cast<float>(e) * (static_cast<float>(G) / static_cast<float>(T)));
  g = g < 0 ? 0 : (g > G - 1 ? G - 1 : g);
  const int64_t lim = (e + 1) * static_cast<int64_t>(G);
  while (g + 1 < G && T * (g + 1) < lim) ++g;
  while (g > 0 && !(T * g < lim)) --g;
  return g;
}

// One row's share of a CTA's element range, and how it is copied.
struct Piece {
  const uint8_t* rowp;
  int row;
  int j0, j1;               // elements [j0, j1) of the row
  uintptr_t lo, hi;         // their bytes
  uintptr_t cp_lo, cp_hi;   // 16-byte-aligned bytes copied by TMA (empty if equal)
  int nst;                  // stages
  int head_end;             // scalar elements [j0, head_end)
  int tail_begin;           // scalar elements [tail_begin, j1)
};

template <int ES>
__device__ __forceinline__ Piece make_piece(const RowStatsArgs& a, int64_t e, int64_t e_end) {
  Piece p;
  p.row = static_cast<int>(e / a.V);
  p.j0 = static_cast<int>(e - static_cast<int64_t>(p.row) * a.V);
  p.j1 = static_cast<int>(min(static_cast<int64_t>(a.V), e_end - static_cast<int64_t>(p.row) * a.V));
  const bool first = p.row < a.set0.rows;
  const RowSet& rs = first ? a.set0 : a.set1;
  const int lr = first ? p.row : p.row - a.set0.rows;
  p.rowp = rs.base + static_cast<int64_t>(lr) * rs.stride_bytes;
  p.lo = reinterpret_cast<uintptr_t>(p.rowp) + static_cast<uintptr_t>(p.j0) * ES;
  p.hi = reinterpret_cast<uintptr_t>(p.rowp) + static_cast<uintptr_t>(p.j1) * ES;
  uintptr_t clo = p.lo & ~static_cast<uintptr_t>(15);
  if (clo < rs.safe_lo) clo = (p.lo + 15) & ~static_cast<uintptr_t>(15);
  uintptr_t chi = (p.hi + 15) & ~static_cast<uintptr_t>(15);
  if (chi > rs.safe_hi) chi = p.hi & ~static_cast<uintptr_t>(15);
  if (chi <= clo) {
    p.cp_lo = p.cp_hi = 0;
    p.nst = 0;
    p.head_end = p.j1;
    p.tail_begin = p.j1;
  } else {
    p.cp_lo = clo;
    p.cp_hi = chi;
    p.nst = static_cast<int>((chi - clo + kK1StageBytes - 1) / kK1StageBytes);
    p.head_end = clo > p.lo ? p.j0 + static_cast<int>((clo - p.lo) / ES) : p.j0;
    p.tail_begin = chi < p.hi ? p.j1 - static_cast<int>((p.hi - chi) / ES) : p.j1;
  }
  return p;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Where a thread's running maximum first appeared: a scalar element (base == 0,
// exact index j) or a stage group (re-read at the end of the piece).
struct GroupCand {
  uintptr_t base;   // global address of the stage's first copied byte, or 0
  int jbase;        // row index of the stage's first element
  int nvec;         // vectors in the stage
  int j;            // exact index of a scalar candidate
};

// Scalar fold (ragged edges only); strict '>' since a thread visits its
// elements in increasing index order.
__device__ __forceinline__ void fold_scalar(float x, int j, float c, float& m, float& mc, float& s,
                                            GroupCand& cand) {
  if (x > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2((m - x) * c);
    m = x;
    mc = x * c;
    cand.base = 0;
    cand.j = j;
  }
  if (x > -INFINITY) s += ex2(fmaf(x, c, -mc));
}

// Fold one thread's unpacked group of a stage into (m, s): at most one
// rescale per group; the argmax keeps only the group where the maximum first
// rose (groups arrive in increasing index order, so a strict '>' keeps the
// lowest index).
template <int N>
__device__ __forceinline__ void fold_values(const float (&f)[kGroupVecs][N], int jbase, int nvec,
                                            uintptr_t gbase, float c, float& m, float& mc, float& s,
                                            GroupCand& cand) {
  float gm[kGroupVecs];
#pragma unroll
  for (int k = 0; k < kGroupVecs; ++k) {
    if constexpr (N == 8)
      gm[k] = fmaxf(max3f(f[k][0], f[k][1], f[k][2]),
                    max3f(max3f(f[k][3], f[k][4], f[k][5]), f[k][6], f[k][7]));
    else
      gm[k] = max3f(f[k][0], f[k][1], fmaxf(f[k][2], f[k][3]));
  }
  const float gmax = fmaxf(max3f(gm[0], gm[1], gm[2]), gm[3]);
  if (gmax > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2((m - gmax) * c);
    m = gmax;
    mc = gmax * c;
    cand.base = gbase;
    cand.jbase = jbase;
    cand.nvec = nvec;
  }
  if (gmax > -INFINITY) {
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int k = 0; k < kGroupVecs; ++k) {
#pragma unroll
      for (int e = 0; e < N; e += 2) {
        acc0 += ex2(fmaf(f[k][e], c, -mc));
        acc1 += ex2(fmaf(f[k][e + 1], c, -mc));
      }
    }
    s += acc0 + acc1;
  }
}

// A full interior stage: four vectors per thread, no masking.
template <int ES>
__device__ __forceinline__ void fold_stage_full(const uint4* sv4, int ct, int jbase, uintptr_t gbase,
                                                float c, float& m, float& mc, float& s, GroupCand& cand) {
  constexpr int N = Elem<ES>::kVec;
  float f[kGroupVecs][N];
#pragma unroll
  for (int k = 0; k < kGroupVecs; ++k) Elem<ES>::unpack(sv4[ct + k * kK1ConsumerThreads], f[k]);
  fold_values<N>(f, jbase, kGroupVecs * kK1ConsumerThreads, gbase, c, m, mc, s, cand);
}

// A short stage, or one holding bytes outside the piece: guarded loads and
// masking. Kept out of line so the full-stage path stays free of them.
template <int ES>
__device__ __noinline__ void fold_stage_edge(const uint4* sv4, int nvec, int ct, int jbase, int j0,
                                             int j1, uintptr_t gbase, float c, float& m, float& mc,
                                             float& s, GroupCand& cand) {
  constexpr int N = Elem<ES>::kVec;
  float f[kGroupVecs][N];
#pragma unroll
  for (int k = 0; k < kGroupVecs; ++k) {
    const int v = ct + k * kK1ConsumerThreads;
    if (v < nvec) {
      Elem<ES>::unpack(sv4[v], f[k]);
    } else {
#pragma unroll
      for (int e = 0; e < N; ++e) f[k][e] = -INFINITY;
    }
    const int jv = jbase + v * N;
#pragma unroll
    for (int e = 0; e < N; ++e)
      if (jv + e < j0 || jv + e >= j1) f[k][e] = -INFINITY;
  }
  fold_values<N>(f, jbase, nvec, gbase, c, m, mc, s, cand);
}

// Lowest index in [j0, j1) of the remembered candidate holding the value m,
// re-read from global memory (INT_MAX if m is -inf).
template <int ES>
__device__ __forceinline__ int resolve_cand(const GroupCand& cand, int ct, float m, int j0, int j1) {
  if (!(m > -INFINITY)) return INT_MAX;
  if (cand.base == 0) return cand.j;
  constexpr int N = Elem<ES>::kVec;
#pragma unroll
  for (int k = 0; k < kGroupVecs; ++k) {
    const int v = ct + k * kK1ConsumerThreads;
    if (v < cand.nvec) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(cand.base) + v);
      float f[N];
      Elem<ES>::unpack(w, f);
      const int jv = cand.jbase + v * N;
#pragma unroll
      for (int e = 0; e < N; ++e)
        if (f[e] == m && jv + e >= j0 && jv + e < j1) return jv + e;
    }
  }
  return INT_MAX;
}

template <int ES>
__global__ void __launch_bounds__(kK1Threads, kK1CtasPerSm) row_stats_kernel(const RowStatsArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kK1Stages];
  __shared__ __align__(8) uint64_t empty_bar[kK1Stages];
  __shared__ float red_m[2][kK1Consumers];
  __shared__ float red_s[2][kK1Consumers];
  __shared__ int red_i[2][kK1Consumers];
  __shared__ int red_e[2][kK1Consumers];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;
  const int64_t E0 = a.T * g / a.G;
  const int64_t E1 = a.T * (g + 1) / a.G;

  // Inputs may come from the kernel before this one, and the partials this
  // kernel writes may still be read by the previous call: wait for it first.
  grid_dep_wait();
  grid_dep_launch();

  if (tid == 0) {
    for (int i = 0; i < kK1Stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kK1Consumers);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0;
      bool ok = true;
      for (int64_t e = E0; e < E1 && ok;) {
        const Piece p = make_piece<ES>(a, e, E1);
        for (int s = 0; s < p.nst; ++s, ++st) {
          const int slot = st % kK1Stages;
          const int use = st / kK1Stages;
          if (use > 0 && !mbar_wait_bounded(smem_u32(&empty_bar[slot]), (use - 1) & 1)) {
            ok = false;
            break;
          }
          const uint32_t off = static_cast<uint32_t>(s) * kK1StageBytes;
          const uint32_t bytes = min(static_cast<uint32_t>(kK1StageBytes),
                                     static_cast<uint32_t>(p.cp_hi - p.cp_lo) - off);
          const uint32_t fb = smem_u32(&full_bar[slot]);
          mbar_arrive_expect_tx(fb, bytes);
          bulk_g2s(smem_u32(ring + slot * kK1StageBytes), reinterpret_cast<const void*>(p.cp_lo + off),
                   bytes, fb);
        }
        e = static_cast<int64_t>(p.row) * a.V + p.j1;
      }
      // The copies still in flight are the last (up to) kK1Stages issued; let
      // them land before the CTA can exit.
      for (int k = max(0, st - kK1Stages); k < st; ++k)
        (void)mbar_wait_bounded(smem_u32(&full_bar[k % kK1Stages]), (k / kK1Stages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ct = tid - 32;
  const int cw = warp - 1;
  const float c = a.c;
  int st = 0, npiece = 0;
  bool ok = true;
  for (int64_t e = E0; e < E1; ++npiece) {
    const Piece p = make_piece<ES>(a, e, E1);
    float m = -INFINITY, mc = -INFINITY, s = 0.f;
    GroupCand cand;
    cand.base = 0;
    cand.jbase = 0;
    cand.nvec = 0;
    cand.j = INT_MAX;
    for (int j = p.j0 + ct; j < p.head_end; j += kK1ConsumerThreads)
      fold_scalar(Elem<ES>::load(p.rowp, j), j, c, m, mc, s, cand);
    for (int sg = 0; sg < p.nst; ++sg, ++st) {
      if (!ok) continue;
      const int slot = st % kK1Stages;
      if (!mbar_wait_bounded(smem_u32(&full_bar[slot]), (st / kK1Stages) & 1)) {
        ok = false;   // stop consuming (and releasing); the producer times out too
        continue;
      }
      const uint32_t off = static_cast<uint32_t>(sg) * kK1StageBytes;
      const int nvec = static_cast<int>(min(static_cast<uintptr_t>(kK1StageBytes), p.cp_hi - p.cp_lo - off) / 16u);
      // row index of the stage's first element (may precede j0 by up to 7)
      const int jbase = p.j0 + static_cast<int>((static_cast<int64_t>(p.cp_lo + off) -
                                                 static_cast<int64_t>(p.lo)) / ES);
      const bool edge = (sg == 0 && p.cp_lo < p.lo) || (sg == p.nst - 1 && p.cp_hi > p.hi);
      const uint4* sv4 = reinterpret_cast<const uint4*>(ring + slot * kK1StageBytes);
      if (!edge && nvec == kGroupVecs * kK1ConsumerThreads)
        fold_stage_full<ES>(sv4, ct, jbase, p.cp_lo + off, c, m, mc, s, cand);
      else
        fold_stage_edge<ES>(sv4, nvec, ct, jbase, p.j0, p.j1, p.cp_lo + off, c, m, mc, s, cand);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
    }
    for (int j = p.tail_begin + ct; j < p.j1; j += kK1ConsumerThreads)
      fold_scalar(Elem<ES>::load(p.rowp, j), j, c, m, mc, s, cand);

    // Warp: max, the lowest index among lanes holding it, and the sum
    // rescaled to the warp max (fixed shuffle order).
    float wm = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    int widx = (m == wm) ? resolve_cand<ES>(cand, ct, m, p.j0, p.j1) : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) widx = min(widx, __shfl_xor_sync(0xffffffffu, widx, o));
    float ws = (m == -INFINITY) ? 0.f : s * ex2((m - wm) * c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);

    // CTA: the consumer warps' results, double-buffered by piece parity so
    // one named barrier per piece suffices.
    const int buf = npiece & 1;
    if (lane == 0) {
      red_m[buf][cw] = wm;
      red_s[buf][cw] = ws;
      red_i[buf][cw] = widx;
      red_e[buf][cw] = ok ? 0 : 1;
    }
    named_barrier_sync(1, kK1ConsumerThreads);
    if (cw == 0 && lane == 0) {
      float rm = red_m[buf][0], rs = red_s[buf][0];
      int ri = red_i[buf][0], re = red_e[buf][0];
      for (int w = 1; w < kK1Consumers; ++w) {
        merge_stats(rm, rs, ri, red_m[buf][w], red_s[buf][w], red_i[buf][w], c);
        re |= red_e[buf][w];
      }
      Partial out;
      out.m = rm;
      out.s = rs;
      out.idx = ri;
      out.err = re;
      a.partials[static_cast<int64_t>(p.row) + g] = out;
    }
    e = static_cast<int64_t>(p.row) * a.V + p.j1;
  }
}

// Merge one row's partials (one per CTA whose range meets the row), in CTA
// order; the first four are loaded together.
__device__ __forceinline__ void merge_row(const Partial* __restrict__ parts, int64_t row, int V,
                                          int64_t T, int G, float c, float& m, float& s, int& idx,
                                          int& err) {
  m = -INFINITY;
  s = 0.f;
  idx = INT_MAX;
  err = 0;
  const int64_t e0 = row * V;
  const int g_lo = cta_of(e0, T, G);
  const int g_hi = cta_of(e0 + V - 1, T, G);
  Partial v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (g_lo + k <= g_hi) v[k] = parts[row + g_lo + k];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (g_lo + k <= g_hi) {
      merge_stats(m, s, idx, v[k].m, v[k].s, v[k].idx, c);
      err |= v[k].err;
    }
  }
  for (int g = g_lo + 4; g <= g_hi; ++g) {
    const Partial w = parts[row + g];
    merge_stats(m, s, idx, w.m, w.s, w.idx, c);
    err |= w.err;
  }
  if (m == -INFINITY) idx = 0;   // every element is -inf: the lowest index attains the max
}

}  // namespace sv
