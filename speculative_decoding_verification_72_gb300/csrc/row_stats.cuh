// K1: fused row-streaming pass. Each CTA owns one segment (<= 32 KB) of one
// logit row. One thread issues the segment's 16-byte-aligned middle as up to
// four 1-D bulk copies (TMA) into shared memory, all in flight at once; the
// ragged head and tail (rows need not start on a 16-byte boundary) are read
// with scalar loads while the copies land. Every thread then folds its
// 16-byte vectors into a running (max, argmax, sum 2^((x - max) c)) as each
// stage's mbarrier completes, and the CTA reduces to one Partial.
//
// This is the single pass over the verify logits that greedy verification
// (argmax, mini-sglang PR #134 verify.py) and the stochastic rules (p(t) and
// q(t) need each row's log-sum-exp, spec-decode README "How it works") share.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kK1Threads = 256;
constexpr int kK1StageBytes = 8192;
constexpr int kK1MaxStages = 4;
constexpr int kK1SegBytes = kK1StageBytes * kK1MaxStages;  // 32 KB per CTA

struct RowSet {
  const uint8_t* base;   // first row
  int64_t stride_bytes;  // row pitch
  int32_t rows;
};

struct RowStatsArgs {
  RowSet set0;         // target rows
  RowSet set1;         // draft rows (rows = 0 if none)
  int32_t V;
  int32_t S;           // segments per row
  int32_t seg_elems;   // elements per segment, a multiple of 64
  float c;             // log2(e) / T
  Partial* partials;   // [(set0.rows + set1.rows) * S]
};

// Scalar fold with full (value, index) ordering: used for the head and tail,
// which are visited out of index order relative to the vector body.
__device__ __forceinline__ void fold_scalar(float x, int j, float c, float& m, float& mc, float& s,
                                            int& idx) {
  if (x > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2((m - x) * c);
    m = x;
    mc = x * c;
    idx = j;
  } else if (x == m && j < idx) {
    idx = j;
  }
  if (x > -INFINITY) s += ex2(fmaf(x, c, -mc));
}

// Vector fold. Within one thread the vectors arrive in increasing index
// order, so a strict '>' keeps the lowest index of the maximum.
template <int ES>
__device__ __forceinline__ void fold_vec(const uint4& w, int j0, float c, float& m, float& mc,
                                         float& s, int& idx) {
  constexpr int N = Elem<ES>::kVec;
  float f[N];
  Elem<ES>::unpack(w, f);
  float vmax = f[0];
#pragma unroll
  for (int k = 1; k < N; ++k) vmax = fmaxf(vmax, f[k]);
  if (vmax > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2((m - vmax) * c);
    int k0 = N - 1;
#pragma unroll
    for (int k = N - 1; k >= 0; --k)
      if (f[k] == vmax) k0 = k;
    idx = j0 + k0;
    m = vmax;
    mc = vmax * c;
  }
  if (vmax > -INFINITY) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < N; ++k) a += ex2(fmaf(f[k], c, -mc));
    s += a;
  }
}

template <int ES>
__global__ void __launch_bounds__(kK1Threads) row_stats_kernel(const RowStatsArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kK1MaxStages];
  __shared__ float red_m[kK1Threads / 32];
  __shared__ float red_s[kK1Threads / 32];
  __shared__ int red_i[kK1Threads / 32];
  __shared__ int s_err;

  const int tid = threadIdx.x;
  const int item = blockIdx.x;
  const int row = item / a.S;
  const int seg = item - row * a.S;
  const bool first_set = row < a.set0.rows;
  const uint8_t* rowp = first_set
                            ? a.set0.base + static_cast<int64_t>(row) * a.set0.stride_bytes
                            : a.set1.base + static_cast<int64_t>(row - a.set0.rows) * a.set1.stride_bytes;
  const int lo = seg * a.seg_elems;
  const int hi = min(a.V, lo + a.seg_elems);
  const uintptr_t glo = reinterpret_cast<uintptr_t>(rowp) + static_cast<uintptr_t>(lo) * ES;
  const uintptr_t ghi = reinterpret_cast<uintptr_t>(rowp) + static_cast<uintptr_t>(hi) * ES;
  const uintptr_t ga = (glo + 15u) & ~static_cast<uintptr_t>(15u);
  const uintptr_t gb = ghi & ~static_cast<uintptr_t>(15u);
  int mid_lo = hi, mid_hi = hi;
  if (ga < gb) {
    mid_lo = lo + static_cast<int>((ga - glo) / ES);
    mid_hi = lo + static_cast<int>((gb - glo) / ES);
  }
  const uint32_t mid_bytes = static_cast<uint32_t>(mid_hi - mid_lo) * ES;
  const int nst = static_cast<int>((mid_bytes + kK1StageBytes - 1) / kK1StageBytes);

  if (tid == 0) {
    s_err = 0;
    for (int st = 0; st < nst; ++st) mbar_init(smem_u32(&bars[st]), 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < nst; ++st) {
      const uint32_t off = static_cast<uint32_t>(st) * kK1StageBytes;
      const uint32_t bytes = min(static_cast<uint32_t>(kK1StageBytes), mid_bytes - off);
      const uint32_t bar = smem_u32(&bars[st]);
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(smem_u32(smem + off), reinterpret_cast<const void*>(ga + off), bytes, bar);
    }
  }

  const float c = a.c;
  float m = -INFINITY, mc = -INFINITY, s = 0.f;
  int idx = INT_MAX;
  for (int j = lo + tid; j < mid_lo; j += kK1Threads)
    fold_scalar(Elem<ES>::load(rowp, j), j, c, m, mc, s, idx);

  bool ok = true;
  for (int st = 0; st < nst; ++st) {
    if (!mbar_wait_bounded(smem_u32(&bars[st]), 0)) {
      ok = false;
      break;
    }
    const uint32_t off = static_cast<uint32_t>(st) * kK1StageBytes;
    const int nvec = static_cast<int>(min(static_cast<uint32_t>(kK1StageBytes), mid_bytes - off) / 16u);
    const uint4* sv4 = reinterpret_cast<const uint4*>(smem + off);
    const int j0 = mid_lo + static_cast<int>(off / ES);
    for (int v = tid; v < nvec; v += kK1Threads)
      fold_vec<ES>(sv4[v], j0 + v * Elem<ES>::kVec, c, m, mc, s, idx);
  }
  if (!ok) s_err = 1;
  if (!ok) {
    // Give the copies still in flight a bounded chance to land before the
    // CTA's shared memory is released.
    for (int st = 0; st < nst; ++st) (void)mbar_wait_bounded(smem_u32(&bars[st]), 0);
  }

  for (int j = mid_hi + tid; j < hi; j += kK1Threads)
    fold_scalar(Elem<ES>::load(rowp, j), j, c, m, mc, s, idx);

  // Block reduction in a fixed order: lanes, then warps.
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_down_sync(0xffffffffu, m, off);
    const float s2 = __shfl_down_sync(0xffffffffu, s, off);
    const int i2 = __shfl_down_sync(0xffffffffu, idx, off);
    merge_stats(m, s, idx, m2, s2, i2, c);
  }
  const int warp = tid >> 5, lane = tid & 31;
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = s;
    red_i[warp] = idx;
  }
  __syncthreads();
  if (warp == 0) {
    constexpr int NW = kK1Threads / 32;
    m = lane < NW ? red_m[lane] : -INFINITY;
    s = lane < NW ? red_s[lane] : 0.f;
    idx = lane < NW ? red_i[lane] : INT_MAX;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_down_sync(0xffffffffu, m, off);
      const float s2 = __shfl_down_sync(0xffffffffu, s, off);
      const int i2 = __shfl_down_sync(0xffffffffu, idx, off);
      merge_stats(m, s, idx, m2, s2, i2, c);
    }
    if (lane == 0) {
      Partial out;
      out.m = m;
      out.s = s;
      out.idx = idx;
      out.err = s_err;
      a.partials[item] = out;
    }
  }
  grid_dep_launch();
}

}  // namespace sv
