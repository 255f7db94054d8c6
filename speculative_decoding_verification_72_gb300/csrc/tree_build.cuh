// EAGLE-style draft-tree construction, the step before tree verification
// (nanospec README, introduction and bench configurations: EAGLE-3 tree
// speculation, depth 5, topk 4; pruned to a fixed node count).
//
// Draft rows arrive rank-ordered: row 0 is the root's, row
// 1 + (d - 2) * topk + r belongs to the r-th best node of level d - 1. A
// node's score is the cumulative draft log-prob of its path,
// score(child) = score(parent) + log_softmax(y / T)[token].
//
// row_topk_kernel: one CTA per draft row streams it once and produces its
// log-sum-exp and its 8 largest logits (lower index first on ties), i.e. the
// candidate tokens of any node whose row it is.
// tree_select_kernel: one CTA per request expands level by level (the topk
// best nodes of a level, score descending and earlier candidate first on
// ties, each take the topk tokens of their row), keeps the n_nodes - 1 best
// candidates (ancestor-closed: a child's score never exceeds its parent's,
// also in fp32, and the parent was created first) and writes them in BFS
// order (level, then score descending, then creation order).
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kTbMaxK = 8;          // largest topk
constexpr int kTbThreads = 256;
constexpr int kTbMaxCands = 1024;   // topk + (depth - 1) * topk^2
constexpr int kTbBatch = 8;         // 16-byte vectors a thread loads together
constexpr int kTbSelThreads = 256;  // threads per request in tree_select_kernel
// A row is read by ceil(V / kTbPieceElems) CTAs. Splitting vocabulary-sized
// rows further was measured slower (the per-CTA bound and list merge then
// cost as much as the streaming), so typical rows take one CTA.
constexpr int kTbPieceElems = 1 << 20;
constexpr int kTbMaxRows = 1 + (kTbMaxCands - kTbMaxK) / kTbMaxK;   // rows per request: 1 + (depth - 1) topk

struct __align__(16) TopRow {
  float lse2;                 // log2-domain log-sum-exp of y * c
  int32_t bad;                // 1 if the row's maximum is not finite
  int32_t pad0, pad1;
  float val[kTbMaxK];         // largest raw logits, descending
  int32_t idx[kTbMaxK];       // their tokens
};

struct RowTopkArgs {
  const uint8_t* base;
  int64_t stride_bytes;
  int32_t V;
  int32_t P;                  // pieces per row (kTbPieceElems elements each, the last shorter)
  float c;                    // log2(e) / T
  TopRow* out;                // [rows]
};

// (a, ia) ranks before (b, ib): larger value, then lower index.
__device__ __forceinline__ bool tb_before(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// Insert (x, j) into a thread's sorted list; the thread visits indices in
// increasing order, so an equal value goes after the ones it already holds.
__device__ __forceinline__ void tb_insert(float (&v)[kTbMaxK], int (&ix)[kTbMaxK], float x, int j) {
  // (the second test admits -inf logits ahead of the empty slots)
  if (!(x > v[kTbMaxK - 1] || (x == v[kTbMaxK - 1] && j < ix[kTbMaxK - 1]))) return;
  v[kTbMaxK - 1] = x;
  ix[kTbMaxK - 1] = j;
#pragma unroll
  for (int q = kTbMaxK - 1; q > 0; --q) {
    if (tb_before(v[q], ix[q], v[q - 1], ix[q - 1])) {
      const float tv = v[q];
      v[q] = v[q - 1];
      v[q - 1] = tv;
      const int ti = ix[q];
      ix[q] = ix[q - 1];
      ix[q - 1] = ti;
    }
  }
}

// One element outside the vector body (scalar head / tail).
__device__ __forceinline__ void tb_visit(float x, int j, float c, float& m, float& s, float (&v)[kTbMaxK],
                                         int (&ix)[kTbMaxK]) {
  if (x > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2((m - x) * c);
    m = x;
  }
  if (x > -INFINITY) s += ex2(fmaf(x, c, -m * c));
  tb_insert(v, ix, x, j);
}

// One 16-byte vector folded into (m, s): the running max moves once per
// vector and the sum takes one exponential per element. Returns the
// vector's maximum (the caller decides whether it may enter the list).
template <int ES>
__device__ __forceinline__ float tb_vector(const uint4& w, float c, float& m, float& s, float (&f)[Elem<ES>::kVec]) {
  constexpr int N = Elem<ES>::kVec;
  Elem<ES>::unpack(w, f);
  float vm = f[0];
#pragma unroll
  for (int e = 1; e < N; ++e) vm = fmaxf(vm, f[e]);
  // exponentials against the running max from before this vector (they do
  // not wait on vm), in two independent f32x2 chains; moved to vm afterwards
  auto vsum = [&](float ref) {
    const float2 c2 = make_float2(c, c), nr = make_float2(-ref, -ref);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < N; e += 4) {
      const float2 t0 = __ffma2_rn(make_float2(f[e], f[e + 1]), c2, nr);
      acc0 = __fadd2_rn(acc0, make_float2(ex2(t0.x), ex2(t0.y)));
      if (e + 2 < N) {
        const float2 t1 = __ffma2_rn(make_float2(f[e + 2], f[e + 3]), c2, nr);
        acc1 = __fadd2_rn(acc1, make_float2(ex2(t1.x), ex2(t1.y)));
      }
    }
    return (acc0.x + acc0.y) + (acc1.x + acc1.y);
  };
  if (m == -INFINITY) {
    if (vm > -INFINITY) {
      m = vm;
      s = vsum(vm * c);
    }
  } else {
    float vs = vsum(m * c);
    if (vm > m) {
      const float d = (m - vm) * c;
      if (d > -64.f && vs <= FLT_MAX) {
        s = (s + vs) * ex2(d);
      } else {
        s = s * ex2(d) + vsum(vm * c);
      }
      m = vm;
    } else {
      s += vs;
    }
  }
  return vm;
}

// The 8th largest of the CTA's per-thread values x (-inf if fewer than 8 are
// finite). Every thread calls it; scratch holds kTbThreads floats.
__device__ __forceinline__ float tb_block_bound(float x, float* scratch) {
  __shared__ float s_bound;
  __syncthreads();   // scratch may still be read from an earlier use
  scratch[threadIdx.x] = x;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float loc[kTbThreads / 32];
#pragma unroll
    for (int q = 0; q < kTbThreads / 32; ++q) loc[q] = scratch[lane * (kTbThreads / 32) + q];
    float kth = -INFINITY;
    for (int r = 0; r < kTbMaxK; ++r) {   // remove the current maximum 8 times
      float lm = loc[0];
      int lq = 0;
#pragma unroll
      for (int q = 1; q < kTbThreads / 32; ++q)
        if (loc[q] > lm) {
          lm = loc[q];
          lq = q;
        }
      float wm = lm;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
      const unsigned own = __ballot_sync(0xffffffffu, lm == wm);
      if (lane == __ffs(own) - 1) {   // one copy of the maximum leaves
#pragma unroll
        for (int q = 0; q < kTbThreads / 32; ++q)
          if (q == lq) loc[q] = -INFINITY;
      }
      kth = wm;
    }
    if (lane == 0) s_bound = kth;
  }
  __syncthreads();
  return s_bound;
}

template <int ES>
__global__ void __launch_bounds__(kTbThreads, 3) row_topk_kernel(const RowTopkArgs a) {
  __shared__ float sv_[kTbThreads][kTbMaxK];
  __shared__ int si_[kTbThreads][kTbMaxK];
  __shared__ float sm_[kTbThreads], ss_[kTbThreads];
  grid_dep_wait();
  grid_dep_launch();
  const int tid = threadIdx.x;
  // this CTA's piece: elements [j_lo, j_lo + Vp) of row blockIdx.x / P
  const int rowi = blockIdx.x / a.P;
  const int piece = blockIdx.x - rowi * a.P;
  const int j_lo = piece * kTbPieceElems;
  const int Vp = min(kTbPieceElems, a.V - j_lo);
  const uint8_t* row = a.base + static_cast<int64_t>(rowi) * a.stride_bytes + static_cast<int64_t>(j_lo) * ES;
  const float c = a.c;
  float m = -INFINITY, s = 0.f;
  float v[kTbMaxK];
  int ix[kTbMaxK];
#pragma unroll
  for (int q = 0; q < kTbMaxK; ++q) {
    v[q] = -INFINITY;
    ix[q] = INT_MAX;
  }
  constexpr int N = Elem<ES>::kVec;
  // 16-byte body [h, h + nv * N) when the row start allows it; the rest scalar
  const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(row) & 15u) / ES);
  const int h = mis ? min(Vp, N - mis) : 0;
  const int nv = (Vp - h) / N;
  // scalar head first, so every thread visits its indices in increasing order
  for (int j = tid; j < h; j += kTbThreads) tb_visit(Elem<ES>::load(row, j), j_lo + j, c, m, s, v, ix);
  const uint4* body = reinterpret_cast<const uint4*>(row + static_cast<int64_t>(h) * ES);
  // After the first batch, `bound` = the 8th largest of the threads' maxima so
  // far: at least 8 elements of the row are >= it, so an element below it is
  // outranked by 8 others and can never enter the row's top 8. Vectors whose
  // maximum is below it skip the list entirely.
  uint4 w[kTbBatch];
  float vmx[kTbBatch];
  // load kTbBatch vectors, fold them into (m, s) and note each one's maximum
  auto load_fold = [&](int q0) {
#pragma unroll
    for (int u = 0; u < kTbBatch; ++u)
      w[u] = (q0 + u * kTbThreads < nv) ? __ldg(body + q0 + u * kTbThreads) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < kTbBatch; ++u) {
      vmx[u] = -INFINITY;
      if (q0 + u * kTbThreads < nv) {
        float f[N];
        vmx[u] = tb_vector<ES>(w[u], c, m, s, f);
      }
    }
  };
  // the vectors that may enter the list, element by element (one copy of the insertion)
  auto insert = [&](int q0, float bound) {
    unsigned pend = 0;
#pragma unroll
    for (int u = 0; u < kTbBatch; ++u)
      if (q0 + u * kTbThreads < nv && vmx[u] >= bound &&
          (vmx[u] > v[kTbMaxK - 1] || ix[kTbMaxK - 1] == INT_MAX))
        pend |= 1u << u;
#pragma unroll 1
    while (pend) {
      const int u = __ffs(pend) - 1;
      pend &= pend - 1;
      uint4 wu = w[0];
#pragma unroll
      for (int q = 1; q < kTbBatch; ++q) wu = (u == q) ? w[q] : wu;
      float f[N];
      Elem<ES>::unpack(wu, f);
      const int j0 = j_lo + h + (q0 + u * kTbThreads) * N;
#pragma unroll 1
      for (int e = 0; e < N; ++e) {
        float fe = f[0];
#pragma unroll
        for (int q = 1; q < N; ++q) fe = (e == q) ? f[q] : fe;
        tb_insert(v, ix, fe, j0 + e);
      }
    }
  };
  // After the first batch is folded, `bound` = the 8th largest of the threads'
  // maxima: at least 8 elements of the row are >= it, so an element below it
  // is outranked by 8 others and can never enter the row's top 8. Only
  // vectors whose maximum reaches it are inserted, the first batch included.
  if (tid < nv) load_fold(tid);
  const float bound = tb_block_bound(m, sm_);   // every thread, outside any loop
  if (tid < nv) insert(tid, bound);
  for (int q0 = tid + kTbBatch * kTbThreads; q0 < nv; q0 += kTbBatch * kTbThreads) {
    load_fold(q0);
    insert(q0, bound);
  }
  for (int j = h + nv * N + tid; j < Vp; j += kTbThreads) tb_visit(Elem<ES>::load(row, j), j_lo + j, c, m, s, v, ix);

  // block merge: pairwise, fixed tree (the order among threads does not matter
  // for the lists: ties are broken by index)
#pragma unroll
  for (int q = 0; q < kTbMaxK; ++q) {
    sv_[tid][q] = v[q];
    si_[tid][q] = ix[q];
  }
  sm_[tid] = m;
  ss_[tid] = s;
  for (int half = kTbThreads / 2; half > 0; half >>= 1) {
    __syncthreads();
    if (tid < half) {
      const int o = tid + half;
      float rv[kTbMaxK];
      int ri[kTbMaxK];
      int pa = 0, pb = 0;
#pragma unroll
      for (int q = 0; q < kTbMaxK; ++q) {   // merge two sorted lists, keep the first 8
        const float av = pa < kTbMaxK ? sv_[tid][pa] : -INFINITY;
        const int ai = pa < kTbMaxK ? si_[tid][pa] : INT_MAX;
        const float bv = pb < kTbMaxK ? sv_[o][pb] : -INFINITY;
        const int bi = pb < kTbMaxK ? si_[o][pb] : INT_MAX;
        const bool takeA = tb_before(av, ai, bv, bi);
        rv[q] = takeA ? av : bv;
        ri[q] = takeA ? ai : bi;
        pa += takeA ? 1 : 0;
        pb += takeA ? 0 : 1;
      }
      float mm = sm_[tid], ssum = ss_[tid];
      const float m2 = sm_[o], s2 = ss_[o];
      if (m2 > mm) {
        ssum = (mm == -INFINITY ? 0.f : ssum * ex2((mm - m2) * c)) + s2;
        mm = m2;
      } else if (m2 != -INFINITY) {
        ssum += s2 * ex2((m2 - mm) * c);
      }
#pragma unroll
      for (int q = 0; q < kTbMaxK; ++q) {
        sv_[tid][q] = rv[q];
        si_[tid][q] = ri[q];
      }
      sm_[tid] = mm;
      ss_[tid] = ssum;
    }
  }
  __syncthreads();
  if (tid == 0) {
    TopRow r;
    const float mm = sm_[0];
    r.bad = !(fabsf(mm) <= FLT_MAX) ? 1 : 0;
    r.lse2 = mm * c + log2f(ss_[0]);
    r.pad0 = r.pad1 = 0;
#pragma unroll
    for (int q = 0; q < kTbMaxK; ++q) {
      r.val[q] = sv_[0][q];
      r.idx[q] = si_[0][q];
    }
    a.out[blockIdx.x] = r;
  }
}

struct TreeSelectArgs {
  const TopRow* rows;     // [B * R * P]: one record per (row, piece)
  int32_t R, P, depth, topk, n_nodes;
  float c;                // log2(e) / T
  int32_t* out_tokens;    // [B, n_nodes]
  int32_t* out_parents;   // [B, n_nodes]
  float* out_scores;      // [B, n_nodes] or nullptr
  int32_t* out_status;    // [B] or nullptr
};

// Rank of candidate i among n candidates by (score desc, creation asc).
__device__ __forceinline__ int tb_rank(const float* sc, const int* ids, int n, int i) {
  int r = 0;
  const float si = sc[ids[i]];
  for (int k = 0; k < n; ++k) {
    const float sk = sc[ids[k]];
    r += (sk > si || (sk == si && ids[k] < ids[i])) ? 1 : 0;
  }
  return r;
}

__global__ void __launch_bounds__(kTbSelThreads) tree_select_kernel(const TreeSelectArgs a) {
  __shared__ float sc[kTbMaxCands];
  __shared__ int par[kTbMaxCands], tok[kTbMaxCands], dep[kTbMaxCands], pos[kTbMaxCands];
  __shared__ int lvl[kTbMaxK * kTbMaxK], front[kTbMaxK], all_ids[kTbMaxCands];
  __shared__ TopRow rows[kTbMaxRows];
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, lane = threadIdx.x;
  const int k = a.topk;
  const float ln2 = kLn2;
  int bad = 0;
  // merge each row's piece records: top 8 by (value desc, index asc), and the
  // log-sum-exps (pieces in order, fixed)
  for (int r = lane; r < a.R; r += kTbSelThreads) {
    const TopRow* pr = a.rows + (static_cast<int64_t>(b) * a.R + r) * a.P;
    TopRow out = pr[0];
    for (int p = 1; p < a.P; ++p) {
      const TopRow q = pr[p];
      float rv[kTbMaxK];
      int ri[kTbMaxK];
      int pa = 0, pb = 0;
#pragma unroll
      for (int t = 0; t < kTbMaxK; ++t) {
        const float av = pa < kTbMaxK ? out.val[pa] : -INFINITY;
        const int ai = pa < kTbMaxK ? out.idx[pa] : INT_MAX;
        const float bv = pb < kTbMaxK ? q.val[pb] : -INFINITY;
        const int bi = pb < kTbMaxK ? q.idx[pb] : INT_MAX;
        const bool takeA = tb_before(av, ai, bv, bi);
        rv[t] = takeA ? av : bv;
        ri[t] = takeA ? ai : bi;
        pa += takeA ? 1 : 0;
        pb += takeA ? 0 : 1;
      }
#pragma unroll
      for (int t = 0; t < kTbMaxK; ++t) {
        out.val[t] = rv[t];
        out.idx[t] = ri[t];
      }
      const float hi = fmaxf(out.lse2, q.lse2);
      out.lse2 = hi == -INFINITY ? -INFINITY : hi + log2f(ex2(out.lse2 - hi) + ex2(q.lse2 - hi));
    }
    out.bad = !(fabsf(out.val[0]) <= FLT_MAX) ? 1 : 0;   // the row's maximum
    rows[r] = out;
  }
  __syncthreads();
  // level 1: the root row's top tokens
  if (lane < k) {
    const TopRow& r0 = rows[0];
    // log-probs are <= 0 (clamped: fp32 rounding must not let a child outscore its parent)
    sc[lane] = fminf(0.f, (r0.val[lane] * a.c - r0.lse2) * ln2);
    par[lane] = -1;
    tok[lane] = r0.idx[lane];
    dep[lane] = 1;
    lvl[lane] = lane;
  }
  if (lane == 0) bad |= rows[0].bad;
  int n = k, lvl_n = k;
  __syncthreads();
  for (int d = 2; d <= a.depth; ++d) {
    // the level's best k nodes, in rank order
    for (int i = lane; i < lvl_n; i += kTbSelThreads) {
      const int r = tb_rank(sc, lvl, lvl_n, i);
      if (r < k) front[r] = lvl[i];
    }
    __syncthreads();
    for (int t = lane; t < k * k; t += kTbSelThreads) {
      const int r = t / k, j = t - r * k;
      const int node = front[r];
      const TopRow& row = rows[1 + (d - 2) * k + r];
      const int cidx = n + t;
      sc[cidx] = sc[node] + fminf(0.f, (row.val[j] * a.c - row.lse2) * ln2);
      par[cidx] = node;
      tok[cidx] = row.idx[j];
      dep[cidx] = d;
      if (j == 0) bad |= row.bad;
    }
    __syncthreads();
    for (int t = lane; t < k * k; t += kTbSelThreads) lvl[t] = n + t;
    n += k * k;
    lvl_n = k * k;
    __syncthreads();
  }
  // keep the n_nodes - 1 best candidates
  for (int i = lane; i < n; i += kTbSelThreads) all_ids[i] = i;
  __syncthreads();
  const int keep = a.n_nodes - 1;
  for (int i = lane; i < n; i += kTbSelThreads) pos[i] = tb_rank(sc, all_ids, n, i) < keep ? 1 : -1;
  __syncthreads();
  // BFS position among the kept: (depth, score desc, creation)
  for (int i = lane; i < n; i += kTbSelThreads) {
    if (pos[i] < 0) continue;
    int p = 1;
    for (int q = 0; q < n; ++q) {
      if (pos[q] < 0) continue;
      const bool before = dep[q] < dep[i] || (dep[q] == dep[i] && (sc[q] > sc[i] || (sc[q] == sc[i] && q < i)));
      p += before ? 1 : 0;
    }
    pos[i] = p + 1000000;   // marked: BFS position + offset (kept)
  }
  __syncthreads();
  const int64_t ob = static_cast<int64_t>(b) * a.n_nodes;
  for (int i = lane; i < n; i += kTbSelThreads) {
    if (pos[i] < 1000000) continue;
    const int p = pos[i] - 1000000;
    a.out_tokens[ob + p] = tok[i];
    a.out_parents[ob + p] = par[i] < 0 ? 0 : pos[par[i]] - 1000000;
    if (a.out_scores) a.out_scores[ob + p] = sc[i];
  }
  if (lane == 0) {
    a.out_tokens[ob] = -1;
    a.out_parents[ob] = -1;
    if (a.out_scores) a.out_scores[ob] = 0.f;
  }
  bad = __syncthreads_or(bad);
  if (lane == 0 && a.out_status) a.out_status[b] = bad ? 4 : 0;   // NONFINITE_ROW
}

}  // namespace sv
