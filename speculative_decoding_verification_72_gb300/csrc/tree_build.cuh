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
// candidate tokens of any node whose row it is. The CTA is warp-specialized
// like the verify pass: warp 0's lane 0 copies the row's 16-byte-aligned hull
// into a 3-stage shared-memory ring with 1-D bulk copies (TMA); 7 consumer
// warps fold each stage into (max, sum of exponentials) and keep per-thread
// top-8 lists. After the first stage the consumers agree on a bound (8
// elements of the row reach it: see tb_bound), which each warp raises again
// after later stages as the maxima cover more of the row; only vectors whose
// maximum reaches it are inserted.
// tree_select_kernel: one CTA per request expands level by level (the topk
// best nodes of a level, score descending and earlier candidate first on
// ties, each take the topk tokens of their row), keeps the n_nodes - 1 best
// candidates (ancestor-closed: a child's score never exceeds its parent's,
// also in fp32, and the parent was created first) and writes them in BFS
// order (level, then score descending, then creation order).
#pragma once

#include "row_stats.cuh"
#include "sv_common.cuh"

namespace sv {

constexpr int kTbMaxK = 8;          // largest topk
constexpr int kTbThreads = 256;
constexpr int kTbConsumers = 7;     // consumer warps of row_topk_kernel (warp 0 copies)
constexpr int kTbConsumerThreads = 32 * kTbConsumers;
constexpr int kTbStageVecs = 8;     // 16-byte vectors per consumer thread per stage
constexpr int kTbStageBytes = kTbConsumerThreads * kTbStageVecs * 16;   // 28 KB
constexpr int kTbStages = 3;
constexpr int kTbSmemBytes = kTbStages * kTbStageBytes;
constexpr int kTbCtasPerSm = 2;
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
  int32_t err;                // 1 if a bounded wait in the producing CTA gave up
  int32_t pad1;
  float val[kTbMaxK];         // largest raw logits, descending
  int32_t idx[kTbMaxK];       // their tokens
};

struct RowTopkArgs {
  const uint8_t* base;
  int64_t stride_bytes;
  uintptr_t safe_lo, safe_hi;   // bytes the caller's buffer holds
  int32_t V;
  int32_t P;                  // pieces per row (kTbPieceElems elements each, the last shorter)
  float c;                    // log2(e) / T
  TopRow* out;                // [rows]
};

// (a, ia) ranks before (b, ib): larger value, then lower index.
__device__ __forceinline__ bool tb_before(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// Fold the statistics (m2, s2) into (m, s), both sums relative to their own
// maximum: the larger maximum stays and the other sum is rescaled to it.
__device__ __forceinline__ void tb_merge_ms(float& m, float& s, float m2, float s2, float c) {
  if (m2 > m) {
    s = (m == -INFINITY ? 0.f : s * ex2((m - m2) * c)) + s2;
    m = m2;
  } else if (m2 != -INFINITY) {
    s += s2 * ex2((m2 - m) * c);
  }
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

// A lower bound on the row's 8th largest value from the consumer threads'
// running maxima (distinct elements, each only rising). Each consumer warp
// publishes the two largest of its lanes' maxima in slot[2 cw], slot[2 cw + 1];
// the bound is the 8th largest of the 2 * kTbConsumers published values, read
// once per warp (lane l loads slot l) and shared by shuffles, so the warp
// agrees on one snapshot. Any mix of older and newer slot values is still a
// set of element values, so the result never exceeds the row's 8th largest:
// warps need not wait for each other (with sync, a consumer barrier between
// publishing and reading makes every warp's current values count).
constexpr int kTbSlots = 2 * kTbConsumers;
static_assert(kTbSlots >= kTbMaxK && kTbSlots <= 32, "one slot per lane");

__device__ __forceinline__ float tb_slots_kth(volatile float* slot, int lane) {
  const float x = lane < kTbSlots ? slot[lane] : -INFINITY;
  int r = 0;   // rank of (x, lane) by value desc, lane asc
#pragma unroll
  for (int q = 0; q < kTbSlots; ++q) {
    const float y = __shfl_sync(0xffffffffu, x, q);
    r += (y > x || (y == x && q < lane)) ? 1 : 0;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < kTbSlots && r == kTbMaxK - 1);
  return __shfl_sync(0xffffffffu, x, __ffs(hit) - 1);
}

__device__ __forceinline__ void tb_publish_top2(float m, int cw, int lane, volatile float* slot) {
  float t1 = m, t2 = -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float o1 = __shfl_xor_sync(0xffffffffu, t1, o);
    const float o2 = __shfl_xor_sync(0xffffffffu, t2, o);
    t2 = fmaxf(fminf(t1, o1), fmaxf(t2, o2));
    t1 = fmaxf(t1, o1);
  }
  if (lane == 0) {
    slot[2 * cw] = t1;
    slot[2 * cw + 1] = t2;
  }
}

__device__ __forceinline__ float tb_bound(float m, int cw, int lane, volatile float* slot, bool sync) {
  tb_publish_top2(m, cw, lane, slot);
  if (sync) named_barrier_sync(1, kTbConsumerThreads);
  else __syncwarp();
  return tb_slots_kth(slot, lane);
}

// One element outside the copied hull: folded into (m, s) with s relative to
// the reference mc (= m c once m is finite, as in the verify pass) and
// offered to the list.
__device__ __forceinline__ void tb_visit_ref(float x, int j, float c, float& m, float& mc, float& s,
                                             float (&v)[kTbMaxK], int (&ix)[kTbMaxK]) {
  if (x > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2(mc - x * c);
    m = x;
    mc = x * c;
  }
  if (x > -INFINITY) s += ex2(fmaf(x, c, -mc));
  tb_insert(v, ix, x, j);
}

// Maximum of one 16-byte vector from its packed words.
template <int ES>
__device__ __forceinline__ float tb_vec_max(const uint4& q) {
  if constexpr (ES == 2) {
    const uint32_t a = max_bf16x2(max_bf16x2(q.x, q.y), max_bf16x2(q.z, q.w));
    return fmaxf(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
  } else {
    return fmaxf(max3f(__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z)), __uint_as_float(q.w));
  }
}

// Offer the elements of half h of this thread's share of a stage that reach
// the bound to the list (vectors ct + (4h + k) * kTbConsumerThreads),
// skipping those outside the piece [0, Vp). A half is offered when its
// maximum reaches the bound, which is rare per thread but frequent per warp,
// so the path first narrows to the vectors, then the elements, that reach it.
template <int ES>
__device__ __forceinline__ void tb_offer_half(const uint4* sv4, int ct, int h, int jbase, int Vp, int j_lo,
                                              float bound, float (&v)[kTbMaxK], int (&ix)[kTbMaxK]) {
  constexpr int N = Elem<ES>::kVec;
#pragma unroll
  for (int k = 0; k < kGroupVecs; ++k) {
    const int vi = ct + (h * kGroupVecs + k) * kTbConsumerThreads;
    const uint4 q4 = sv4[vi];
    if (!(tb_vec_max<ES>(q4) >= bound)) continue;   // packed maximum first
    float f[N];
    Elem<ES>::unpack(q4, f);
    const int jv = jbase + vi * N;
    unsigned cand = 0u;
#pragma unroll
    for (int e = 0; e < N; ++e)
      if (f[e] >= bound && jv + e >= 0 && jv + e < Vp) cand |= 1u << e;
#pragma unroll 1
    while (cand) {
      const int e = __ffs(cand) - 1;
      cand &= cand - 1u;
      float fe = f[0];
#pragma unroll
      for (int q = 1; q < N; ++q) fe = (e == q) ? f[q] : fe;
      tb_insert(v, ix, fe, j_lo + jv + e);
    }
  }
}

template <int ES>
__global__ void __launch_bounds__(kTbThreads, kTbCtasPerSm) row_topk_kernel(const RowTopkArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kTbStages];
  __shared__ __align__(8) uint64_t empty_bar[kTbStages];
  __shared__ float sv_[kTbThreads][kTbMaxK];
  __shared__ int si_[kTbThreads][kTbMaxK];
  __shared__ float sm_[kTbThreads], ss_[kTbThreads];
  __shared__ float s_slot[kTbSlots];   // published warp maxima (tb_bound)
  __shared__ int s_err, s_ncand;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {   // shared-memory setup overlaps the previous kernel
    s_err = 0;
    s_ncand = 0;
    for (int q = 0; q < kTbSlots; ++q) s_slot[q] = -INFINITY;
    for (int i = 0; i < kTbStages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kTbConsumers);
    }
    fence_barrier_init();
  }
  // this CTA's piece: elements [j_lo, j_lo + Vp) of row blockIdx.x / P
  const int rowi = blockIdx.x / a.P;
  const int piece = blockIdx.x - rowi * a.P;
  const int j_lo = piece * kTbPieceElems;
  const int Vp = min(kTbPieceElems, a.V - j_lo);
  const uint8_t* row = a.base + static_cast<int64_t>(rowi) * a.stride_bytes + static_cast<int64_t>(j_lo) * ES;
  const float c = a.c;
  // 16-byte hull of the piece, clipped to the buffer; elements it misses are
  // read from global memory (at most 15 bytes at each end)
  const uintptr_t L = reinterpret_cast<uintptr_t>(row);
  const uintptr_t H = L + static_cast<uintptr_t>(Vp) * ES;
  uintptr_t clo = L & ~static_cast<uintptr_t>(15);
  if (clo < a.safe_lo) clo = (L + 15) & ~static_cast<uintptr_t>(15);
  uintptr_t chi = (H + 15) & ~static_cast<uintptr_t>(15);
  if (chi > a.safe_hi) chi = H & ~static_cast<uintptr_t>(15);
  const uint32_t nbytes = chi > clo ? static_cast<uint32_t>(chi - clo) : 0u;
  const int e0 = nbytes ? static_cast<int>((static_cast<int64_t>(clo) - static_cast<int64_t>(L)) / ES) : 0;
  const int nst = static_cast<int>((nbytes + kTbStageBytes - 1) / kTbStageBytes);
  const int c_lo = nbytes ? max(0, e0) : Vp;             // copied piece elements [c_lo, c_hi)
  const int c_hi = nbytes ? min(Vp, e0 + static_cast<int>(nbytes / ES)) : Vp;

  // The first copies' bytes go to L2 before the dependency wait (a prefetch
  // returns nothing to the program; the previous kernel's writes land in L2).
  if (tid == 0)
    for (int st = 0; st < nst && st < kTbStages; ++st)
      bulk_prefetch_l2(reinterpret_cast<const void*>(clo + static_cast<uint32_t>(st) * kTbStageBytes),
                       min(static_cast<uint32_t>(kTbStageBytes), nbytes - static_cast<uint32_t>(st) * kTbStageBytes));
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();

  float m = -INFINITY, s = 0.f;
  float v[kTbMaxK];
  int ix[kTbMaxK];
#pragma unroll
  for (int q = 0; q < kTbMaxK; ++q) {
    v[q] = -INFINITY;
    ix[q] = INT_MAX;
  }
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int slot = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int st = 0; st < nst; ++st, issued = st) {
        if (st >= kTbStages && !mbar_wait_bounded(smem_u32(&empty_bar[slot]), phase ^ 1)) {
          ok = false;
          break;
        }
        const uint32_t off = static_cast<uint32_t>(st) * kTbStageBytes;
        const uint32_t bytes = min(static_cast<uint32_t>(kTbStageBytes), nbytes - off);
        const uint32_t fb = smem_u32(&full_bar[slot]);
        mbar_arrive_expect_tx(fb, bytes);
        bulk_g2s(smem_u32(ring + slot * kTbStageBytes), reinterpret_cast<const void*>(clo + off), bytes, fb);
        if (++slot == kTbStages) {
          slot = 0;
          phase ^= 1;
        }
      }
      if (!ok) atomicOr(&s_err, 1);
      // the copies still in flight (among the last kTbStages issued, also
      // after a wait gave up) land before the CTA exits
      for (int q = max(0, issued - kTbStages); q < issued; ++q)
        (void)mbar_wait_bounded(smem_u32(&full_bar[q % kTbStages]), (q / kTbStages) & 1);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- consumers
    // The verify pass's fold (two 16-word groups per stage, packed max and
    // fp32x2 exponential sums against the reference from before the group),
    // plus the list: a half whose maximum reaches the bound is offered
    // element by element.
    static_assert(kTbStageVecs == 2 * kGroupVecs && kTbConsumerThreads == kK1ConsumerThreads, "verify-pass group layout");
    constexpr int kTbFullVecs = kTbStageVecs * kTbConsumerThreads;
    const int ct = tid - 32;
    float mc = 0.f;   // exponent reference of s
    // the head the copy misses, first: each thread visits its indices in increasing order
    for (int j = ct; j < c_lo; j += kTbConsumerThreads) tb_visit_ref(Elem<ES>::load(row, j), j_lo + j, c, m, mc, s, v, ix);
    float bound = -INFINITY;
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    constexpr int kStageElems = kTbStageBytes / ES;
    for (int st = 0; st < nst; ++st) {
      if (ok && !mbar_wait_bounded(smem_u32(&full_bar[slot]), phase)) {
        ok = false;
        atomicOr(&s_err, 1);
      }
      uint4* sv4 = reinterpret_cast<uint4*>(ring + slot * kTbStageBytes);
      float ga = -INFINITY, gb = -INFINITY;
      const int jbase = e0 + st * kStageElems;   // piece index of the stage's first element
      if (ok) {
        const int nvec = static_cast<int>(min(static_cast<uint32_t>(kTbStageBytes), nbytes - st * kTbStageBytes) / 16);
        const bool first_edge = st == 0 && e0 < 0;
        const bool last_hull = st == nst - 1 && e0 + static_cast<int>(nbytes / ES) > Vp;
        if (first_edge || last_hull || nvec != kTbFullVecs)
          mask_stage<ES, kTbStageVecs>(sv4, ct, nvec, jbase, 0, Vp, first_edge ? 0 : -1, last_hull ? nvec - 1 : -1);
        uint32_t w[kGroupWords];
        load_half(sv4, ct, 0, w);
        const float sa = group_sum<ES>(w, c, mc);
        ga = group_max<ES>(w);
        load_half(sv4, ct, 1, w);
        const float sb = group_sum<ES>(w, c, mc);
        gb = group_max<ES>(w);
        const float gmax = fmaxf(ga, gb);
        const float gsum = sa + sb;
        if (gmax > m) {
          const float nmc = gmax * c;
          const float d = mc - nmc;
          if (gsum <= FLT_MAX && d <= 20.f) {
            s = (s + gsum) * ex2(d);
          } else {
            float r = group_sum<ES>(w, c, nmc);
            load_half(sv4, ct, 0, w);
            r += group_sum<ES>(w, c, nmc);
            s = (m == -INFINITY ? 0.f : s * ex2(d)) + r;
          }
          m = gmax;
          mc = nmc;
        } else if (gmax > -INFINITY) {
          s += gsum;
        }
      }
      // The bound tightens as the maxima cover more of the row (after
      // stages 0, 1, 3, 6: each refresh roughly halves the share of elements
      // that reach it); fewer offers then interrupt the warps.
      if (st == 0 || st == 1 || st == 3 || st == 6) bound = fmaxf(bound, tb_bound(m, ct >> 5, lane, s_slot, st == 0));
      if (ok) {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {   // one copy of the offer path
          const float gh = h ? gb : ga;
          if (gh >= bound && (gh > v[kTbMaxK - 1] || ix[kTbMaxK - 1] == INT_MAX))
            tb_offer_half<ES>(sv4, ct, h, jbase, Vp, j_lo, bound, v, ix);
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
      if (++slot == kTbStages) {
        slot = 0;
        phase ^= 1;
      }
    }
    for (int j = c_hi + ct; j < Vp; j += kTbConsumerThreads) tb_visit_ref(Elem<ES>::load(row, j), j_lo + j, c, m, mc, s, v, ix);
    if (m > -INFINITY) s = s * ex2(mc - m * c);   // s relative to m c for the merge (mc == m c already)
    tb_publish_top2(m, ct >> 5, lane, s_slot);   // final maxima for the gather threshold
  }
  __syncthreads();   // the final maxima are published

  // Row statistics: each warp folds its lanes' (m, s) with shuffles (fixed
  // order), then thread 0 folds the warps' in order.
  float wm = m, wsum = s;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, wm, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, wsum, o);
    tb_merge_ms(wm, wsum, m2, s2, c);
  }
  if (lane == 0) {
    sm_[warp] = wm;
    ss_[warp] = wsum;
  }
  // The row's top 8 hide among the list entries that reach the final bound:
  // the bound never exceeds the row's 8th largest value and every element
  // that reaches it was offered, so each of the top 8 sits in its thread's
  // list. Those entries (a dozen or so; at most every list entry) are
  // gathered, and one warp picks the 8 first by (value desc, index asc).
  float* cv = &sv_[0][0];
  int* ci = &si_[0][0];
  const float fbound = tb_slots_kth(s_slot, lane);   // every warp, same final snapshot
  int nmine = 0;
#pragma unroll
  for (int q = 0; q < kTbMaxK; ++q) nmine += v[q] >= fbound ? 1 : 0;
  if (nmine) {   // (s_ncand was zeroed at the start)
    const int at = atomicAdd(&s_ncand, nmine);
#pragma unroll
    for (int q = 0; q < kTbMaxK; ++q)
      if (q < nmine) {
        cv[at + q] = v[q];
        ci[at + q] = ix[q];
      }
  }
  __syncthreads();
  if (warp == 0 && s_ncand <= 32) {
    // one candidate per lane: its rank by (value desc, index asc) against
    // all others in one pass of shuffles; ranks 0..7 are the top 8 (the
    // bound guarantees at least 8 candidates unless it is -inf, and then every
    // list entry is gathered, more than 32)
    const int n = s_ncand;
    const float x = lane < n ? cv[lane] : -INFINITY;
    const int xi = lane < n ? ci[lane] : INT_MAX;
    int r = 0;
#pragma unroll 8
    for (int q = 0; q < 32; ++q) {
      const float y = __shfl_sync(0xffffffffu, x, q);
      const int yi = __shfl_sync(0xffffffffu, xi, q);
      r += (q < n && q != lane && tb_before(y, yi, x, xi)) ? 1 : 0;
    }
    TopRow* out = a.out + blockIdx.x;
    if (lane < n && r < kTbMaxK) {
      out->val[r] = x;
      out->idx[r] = xi;
    }
    if (lane >= n && lane < kTbMaxK) {   // (fewer than 8 candidates: empty slots)
      out->val[lane] = -INFINITY;
      out->idx[lane] = INT_MAX;
    }
  } else if (warp == 0) {
    // each lane keeps the best 8 of its strided share, then 8 rounds of a
    // warp-wide (value desc, index asc) maximum pop one entry each
    float lv[kTbMaxK];
    int li[kTbMaxK];
#pragma unroll
    for (int q = 0; q < kTbMaxK; ++q) {
      lv[q] = -INFINITY;
      li[q] = INT_MAX;
    }
    const int n = s_ncand;
    for (int k = lane; k < n; k += 32) tb_insert(lv, li, cv[k], ci[k]);
    float outv = -INFINITY;
    int outi = INT_MAX;
    for (int r = 0; r < kTbMaxK; ++r) {
      float bv = lv[0];
      int bi = li[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (tb_before(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (lane == r) {
        outv = bv;
        outi = bi;
      }
      if (li[0] == bi && lv[0] == bv) {   // the owner pops its head (indices are unique)
#pragma unroll
        for (int q = 0; q < kTbMaxK - 1; ++q) {
          lv[q] = lv[q + 1];
          li[q] = li[q + 1];
        }
        lv[kTbMaxK - 1] = -INFINITY;
        li[kTbMaxK - 1] = INT_MAX;
      }
    }
    TopRow* out = a.out + blockIdx.x;
    if (lane < kTbMaxK) {
      out->val[lane] = outv;
      out->idx[lane] = outi;
    }
  } else if (warp == 1 && lane == 0) {   // the row statistics, beside the selection
    float mm = -INFINITY, ssum = 0.f;
    for (int w = 0; w < kTbThreads / 32; ++w) tb_merge_ms(mm, ssum, sm_[w], ss_[w], c);
    TopRow* out = a.out + blockIdx.x;
    out->bad = !(fabsf(mm) <= FLT_MAX) ? 1 : 0;
    out->lse2 = mm * c + log2f(ssum);
    out->err = s_err;
    out->pad1 = 0;
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

__global__ void __launch_bounds__(kTbSelThreads) tree_select_kernel(const TreeSelectArgs a) {
  __shared__ float sc[kTbMaxCands];
  __shared__ int par[kTbMaxCands], tok[kTbMaxCands], dep[kTbMaxCands], pos[kTbMaxCands], bfs[kTbMaxCands];
  __shared__ int s_excl[kTbMaxCands];
  __shared__ int s_nexcl;
  __shared__ int front[kTbMaxK];
  __shared__ TopRow rows[kTbMaxRows];
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, lane = threadIdx.x;
  const int k = a.topk;
  if (lane == 0) s_nexcl = 0;
  const float ln2 = kLn2;
  int bad = 0, err = 0;
  // merge each row's piece records: top 8 by (value desc, index asc), and the
  // log-sum-exps (pieces in order, fixed); rows of one piece are copied as
  // they are, 16 bytes per thread
  static_assert(sizeof(TopRow) % 16 == 0, "row records move as 16-byte words");
  constexpr int kRowWords = sizeof(TopRow) / 16;
  if (a.P == 1) {   // (the row pass set bad from the same maximum)
    static_assert(offsetof(TopRow, err) == 8, "err is the third word of a record's first 16 bytes");
    const uint4* src = reinterpret_cast<const uint4*>(a.rows + static_cast<int64_t>(b) * a.R);
    uint4* dst = reinterpret_cast<uint4*>(rows);
    for (int w = lane; w < a.R * kRowWords; w += kTbSelThreads) {
      const uint4 q = src[w];
      dst[w] = q;
      if (w % kRowWords == 0) err |= static_cast<int>(q.z);
    }
  }
  for (int r = lane; r < a.R && a.P > 1; r += kTbSelThreads) {
    const TopRow* pr = a.rows + (static_cast<int64_t>(b) * a.R + r) * a.P;
    TopRow out = pr[0];
    err |= out.err;
    for (int p = 1; p < a.P; ++p) {
      const TopRow q = pr[p];
      err |= q.err;
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
  // Level 1 is the root row's top tokens. A level's candidates are
  // consecutive: [base, base + lvl_n), creation order. One warp builds the
  // levels (no block barriers): lane l ranks candidates l, l + 32, ... of the
  // level against all of them (score desc, creation asc), then lanes expand
  // the best k, k children each.
  const int wid = lane >> 5, wl = lane & 31;
  const int n = k + (a.depth - 1) * k * k;   // candidates after the last level
  if (wid == 0) {
    if (wl < k) {
      const TopRow& r0 = rows[0];
      // log-probs are <= 0 (clamped: fp32 rounding must not let a child outscore its parent)
      sc[wl] = fminf(0.f, (r0.val[wl] * a.c - r0.lse2) * ln2);
      par[wl] = -1;
      tok[wl] = r0.idx[wl];
      dep[wl] = 1;
    }
    if (wl == 0) bad |= rows[0].bad;
    __syncwarp();
    int nn = k, base = 0, lvl_n = k;
    for (int d = 2; d <= a.depth; ++d) {
      for (int i = wl; i < lvl_n; i += 32) {
        const float si = sc[base + i];
        int r = 0;
#pragma unroll 4
        for (int q = 0; q < lvl_n; ++q) {
          const float sq = sc[base + q];
          r += static_cast<int>((sq > si) | ((sq == si) & (q < i)));
        }
        if (r < k) front[r] = base + i;
      }
      __syncwarp();
      for (int t = wl; t < k * k; t += 32) {
        const int r = t / k, j = t - r * k;
        const int node = front[r];
        const TopRow& row = rows[1 + (d - 2) * k + r];
        const int cidx = nn + t;
        sc[cidx] = sc[node] + fminf(0.f, (row.val[j] * a.c - row.lse2) * ln2);
        par[cidx] = node;
        tok[cidx] = row.idx[j];
        dep[cidx] = d;
        if (j == 0) bad |= row.bad;
      }
      __syncwarp();
      base = nn;
      nn += k * k;
      lvl_n = k * k;
    }
  }
  __syncthreads();
  // Keep the n_nodes - 1 best candidates and give the kept ones their BFS
  // position (depth, score desc, creation), in one pass: thread t takes
  // candidates t, t + blockDim, ... and counts, over all n (broadcast loads,
  // branch-free tests), the candidates ranked before it by score and those
  // before it in BFS order. The excluded ones (the n - keep last by score, a
  // handful) are gathered, and a kept candidate's position is its BFS count
  // less the excluded candidates before it.
  const int keep = a.n_nodes - 1;
  for (int i = lane; i < n; i += kTbSelThreads) {
    const float si = sc[i];
    const int di = dep[i];
    int r = 0, pb = 0;
#pragma unroll 8
    for (int q = 0; q < n; ++q) {
      const float sq = sc[q];
      const int dq = dep[q];
      const bool by_score = (sq > si) | ((sq == si) & (q < i));
      r += static_cast<int>(by_score);
      pb += static_cast<int>((dq < di) | ((dq == di) & by_score));
    }
    const bool kept = r < keep;
    if (!kept) s_excl[atomicAdd(&s_nexcl, 1)] = i;
    pos[i] = kept ? pb : -1;
  }
  __syncthreads();
  const int nexcl = s_nexcl;
  for (int i = lane; i < n; i += kTbSelThreads) {
    int p = pos[i];
    if (p >= 0) {
      const float si = sc[i];
      const int di = dep[i];
      for (int e = 0; e < nexcl; ++e) {
        const int q = s_excl[e];
        const float sq = sc[q];
        const int dq = dep[q];
        p -= static_cast<int>((dq < di) | ((dq == di) & ((sq > si) | ((sq == si) & (q < i)))));
      }
      p += 1;   // position 0 is the root
    }
    bfs[i] = p;
  }
  __syncthreads();
  const int64_t ob = static_cast<int64_t>(b) * a.n_nodes;
  for (int i = lane; i < n; i += kTbSelThreads) {
    const int p = bfs[i];
    if (p < 0) continue;
    a.out_tokens[ob + p] = tok[i];
    a.out_parents[ob + p] = par[i] < 0 ? 0 : bfs[par[i]];
    if (a.out_scores) a.out_scores[ob + p] = sc[i];
  }
  if (lane == 0) {
    a.out_tokens[ob] = -1;
    a.out_parents[ob] = -1;
    if (a.out_scores) a.out_scores[ob] = 0.f;
  }
  bad = __syncthreads_or(bad);
  err = __syncthreads_or(err);
  if (lane == 0 && a.out_status) a.out_status[b] = (bad ? SV_STATUS_NONFINITE_ROW : 0) | (err ? SV_STATUS_TIMEOUT : 0);
}

}  // namespace sv
