// K1: the single streaming pass over the verify logits (argmax for greedy
// verification, mini-sglang PR #134 verify.py; log-sum-exp for p(t) and q(t),
// spec-decode README "How it works").
//
// Persistent and warp-specialized. The rows of both logit sets form one
// flattened element space of T = rows * V elements; CTA g owns the elements
// [T g / G, T (g+1) / G), so every CTA streams the same number of bytes
// whatever the row count. Warp 0 is the producer: one lane walks the CTA's
// row pieces and issues 1-D bulk copies (TMA) of up to 28 KB into a 3-stage
// shared-memory ring, arming each stage's "full" mbarrier with the byte count
// and reusing a stage once all consumer warps have released it on its
// "empty" mbarrier. Warps 1..7 consume: each thread folds its 16-byte
// vectors of each stage into a running (max, sum 2^((x - max) c)) and
// remembers the vector holding its first maximum. At the end of every row
// piece the consumers resolve the exact argmax from a per-thread shared-memory
// stash of that vector (copied when the maximum rose), reduce it within the
// warp and write one Partial per (warp, row piece), so no warp waits for,
// counts or merges another. The decide kernel merges a row's partials.
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

constexpr int kK1Consumers = 7;                       // consumer warps
constexpr int kK1Threads = 32 * (kK1Consumers + 1);   // + one producer warp
constexpr int kK1ConsumerThreads = 32 * kK1Consumers;
constexpr int kK1CtasPerSm = 2;
// Each of an SM's four schedulers holds a quarter of the 64K registers and
// its share of the resident warps: with 2 CTAs of 8 warps every scheduler
// gets 4 warps, which leaves 128 registers per thread.
constexpr int kK1WarpsPerScheduler = (kK1CtasPerSm * (kK1Consumers + 1) + 3) / 4;
constexpr int kK1MaxRegs = (16384 / (kK1WarpsPerScheduler * 32)) / 8 * 8;
// Vectors one consumer thread folds per stage, in halves of kGroupVecs.
constexpr int kStageVecs = 8;
constexpr int kGroupVecs = 4;
constexpr int kStageHalves = kStageVecs / kGroupVecs;
constexpr int kK1StageBytes = kK1ConsumerThreads * kStageVecs * 16;   // 28 KB
constexpr int kK1Stages = 3;
constexpr int kK1RingBytes = kK1StageBytes * kK1Stages;
// Per-thread copy of the 16-byte vector that holds its running maximum.
constexpr int kK1StashBytes = kK1ConsumerThreads * 16;
constexpr int kK1SmemBytes = kK1RingBytes + kK1StashBytes;
constexpr int kK1MaxCtas = 4096;                      // bound used to size the workspace
// Piece-result slots of the early-exit row pass (row_stats_early.cuh), which
// merges a row's warp results in the CTA: warps are at most kK1Stages pieces
// apart when every piece has a copied stage, plus one piece per buffer edge
// handled by scalar loads alone (two per row set, two row sets).
constexpr int kK1RedBufs = 8;
static_assert(kK1RedBufs >= kK1Stages + 5 && (kK1RedBufs & (kK1RedBufs - 1)) == 0, "piece-result ring");
static_assert(kK1Consumers <= 8, "the piece merge reduces lanes 0..7");
constexpr int kK1MinBytesPerCta = 16384;
static_assert(kStageHalves == 1 || kStageHalves == 2, "a stage is folded as one or two groups per thread");

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
  Partial* partials;   // [(rows + G) * kK1Consumers]: slot (row + cta) * kK1Consumers + warp
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

// The piece of row `row` that starts at element j0 and ends at the row's end
// or at flattened element e_end, whichever is first.
template <int ES>
__device__ __forceinline__ Piece make_piece(const RowStatsArgs& a, int row, int j0, int64_t e_end) {
  Piece p;
  p.row = row;
  p.j0 = j0;
  p.j1 = static_cast<int>(min(static_cast<int64_t>(a.V), e_end - static_cast<int64_t>(row) * a.V));
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

// Where a thread's running maximum first appeared: a scalar element
// (stage -1, exact index j) or one 16-byte vector of one stage of the current
// row piece, which the thread has copied to its shared-memory stash.
struct GroupCand {
  int stage;   // stage index within the piece, or -1 for a scalar element
  int vec;     // the vector's k in the thread's stage share (v = ct + k kK1ConsumerThreads)
  int j;       // exact index of a scalar candidate
  int jbase;   // row index of the candidate stage's first element
};

// Scalar fold (ragged edges only); strict '>' since a thread visits its
// elements in increasing index order.
__device__ __forceinline__ void fold_scalar(float x, int j, float c, float& m, float& mc, float& s,
                                            GroupCand& cand) {
  if (x > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2((m - x) * c);
    m = x;
    mc = x * c;
    cand.stage = -1;
    cand.j = j;
  }
  if (x > -INFINITY) s += ex2(fmaf(x, c, -mc));
}

// A group is 16 32-bit words (kGroupVecs vectors): 16 fp32 elements, or 32
// bf16 elements packed two per word (low half first).
constexpr int kGroupWords = kGroupVecs * 4;

__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Maximum of a group (NaN ignored: max.bf16x2 and max.f32 return the other
// operand). vm[k] receives vector k's maximum as computed on the way: for
// bf16 the packed pair max of its 8 elements, for fp32 the float's bits
// (vec_max_of turns either into a float). The vectors' maxima come free from
// the reduction tree, so locating the vector that holds a new maximum needs
// no second pass over the stage.
template <int ES>
__device__ __forceinline__ float group_max(const uint32_t (&w)[kGroupWords], uint32_t (&vm)[kGroupVecs]) {
  if constexpr (ES == 2) {
    uint32_t a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = max_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) vm[i] = max_bf16x2(a[2 * i], a[2 * i + 1]);
    const uint32_t b = max_bf16x2(max_bf16x2(vm[0], vm[1]), max_bf16x2(vm[2], vm[3]));
    return fmaxf(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u));
  } else {
    float t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      t[i] = fmaxf(max3f(__uint_as_float(w[4 * i]), __uint_as_float(w[4 * i + 1]), __uint_as_float(w[4 * i + 2])),
                   __uint_as_float(w[4 * i + 3]));
      vm[i] = __float_as_uint(t[i]);
    }
    return fmaxf(max3f(t[0], t[1], t[2]), t[3]);
  }
}

template <int ES>
__device__ __forceinline__ float vec_max_of(uint32_t vmk) {
  if constexpr (ES == 2)
    return fmaxf(__uint_as_float(vmk << 16), __uint_as_float(vmk & 0xffff0000u));
  else
    return __uint_as_float(vmk);
}

template <int ES>
__device__ __forceinline__ float group_max(const uint32_t (&w)[kGroupWords]) {
  uint32_t vm[kGroupVecs];
  return group_max<ES>(w, vm);
}

// sum over the group of 2^(x c - mc), with packed fp32x2 FMA / add.
template <int ES>
__device__ __forceinline__ float group_sum(const uint32_t (&w)[kGroupWords], float c, float mc) {
  const float2 c2 = make_float2(c, c);
  const float2 nmc2 = make_float2(-mc, -mc);
  float2 acc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
  constexpr int kPairs = ES == 2 ? kGroupWords : kGroupWords / 2;
#pragma unroll
  for (int k = 0; k < kPairs; ++k) {
    float2 x;
    if constexpr (ES == 2) {
      x = make_float2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
    } else {
      x = make_float2(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1]));
    }
    const float2 t = __ffma2_rn(x, c2, nmc2);
    acc[k & 3] = __fadd2_rn(acc[k & 3], make_float2(ex2(t.x), ex2(t.y)));
  }
  const float2 a01 = __fadd2_rn(acc[0], acc[1]);
  const float2 a23 = __fadd2_rn(acc[2], acc[3]);
  const float2 a = __fadd2_rn(a01, a23);
  return a.x + a.y;
}

constexpr int kStageFullVecs = kStageVecs * kK1ConsumerThreads;

// Edge stages (the first and last of a piece whose copy hull reaches past the
// piece, or a short last stage) are masked in place before the fold. Vectors
// past nvec (not written by the copy) become all -inf; each thread rewrites
// only its own such vectors v = ct + k * kK1ConsumerThreads. The elements
// outside [j0, j1) can only sit in vectors mask_lo_v and mask_hi_v (the
// hull's first and last); each is rewritten by the one thread that folds it,
// so the other threads do no per-element work. The fold then has a single
// code path for every stage.
template <int ES>
__device__ __forceinline__ void mask_vec(uint4* sv4, int v, int jbase, int j0, int j1) {
  constexpr int N = Elem<ES>::kVec;
  const uint4 q = sv4[v];
  uint32_t word[4] = {q.x, q.y, q.z, q.w};
  const int jv = jbase + v * N;
#pragma unroll
  for (int e = 0; e < N; ++e) {
    if (jv + e < j0 || jv + e >= j1) {
      if constexpr (ES == 2) {
        const int wi = e >> 1;
        word[wi] = (e & 1) ? ((word[wi] & 0x0000ffffu) | 0xff800000u) : ((word[wi] & 0xffff0000u) | 0x0000ff80u);
      } else {
        word[e] = 0xff800000u;
      }
    }
  }
  sv4[v] = make_uint4(word[0], word[1], word[2], word[3]);
}

template <int ES, int SV = kStageVecs>
__device__ __forceinline__ void mask_stage(uint4* sv4, int ct, int nvec, int jbase, int j0, int j1,
                                           int mask_lo_v, int mask_hi_v, int nh = SV / kGroupVecs) {
  constexpr uint32_t kNegInfWord = ES == 2 ? 0xff80ff80u : 0xff800000u;   // -inf in every element
  if (nvec < SV * kK1ConsumerThreads) {   // a short stage (uniform over the CTA)
#pragma unroll
    for (int k = 0; k < SV; ++k) {
      // a half the warp does not fold (stage_halves) is left as the copy wrote it
      const int v = ct + k * kK1ConsumerThreads;
      if (k < nh * kGroupVecs && v >= nvec) sv4[v] = make_uint4(kNegInfWord, kNegInfWord, kNegInfWord, kNegInfWord);
    }
  }
  if (mask_lo_v >= 0 && ct == mask_lo_v % kK1ConsumerThreads) mask_vec<ES>(sv4, mask_lo_v, jbase, j0, j1);
  if (mask_hi_v >= 0 && mask_hi_v != mask_lo_v && ct == mask_hi_v % kK1ConsumerThreads)
    mask_vec<ES>(sv4, mask_hi_v, jbase, j0, j1);
  // These generic-proxy writes precede the next bulk copy into the slot.
  // (Fencing only in the threads that wrote was measured slower.)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One half (kGroupVecs vectors, 16 words) of a thread's share of a stage:
// vectors v = ct + (4*h + k) * kK1ConsumerThreads.
__device__ __forceinline__ void load_half(const uint4* sv4, int ct, int h, uint32_t (&w)[kGroupWords]) {
#pragma unroll
  for (int k = 0; k < kGroupVecs; ++k) {
    const uint4 q = sv4[ct + (h * kGroupVecs + k) * kK1ConsumerThreads];
    w[4 * k] = q.x;
    w[4 * k + 1] = q.y;
    w[4 * k + 2] = q.z;
    w[4 * k + 3] = q.w;
  }
}

// Record where the thread's new maximum gmax first appears in half h of this
// stage: the lowest vector of the half whose maximum (vm, from group_max)
// equals gmax, copied to the thread's stash slot stash[ct]; resolve_cand
// later finds the element inside it.
template <int ES>
__device__ __forceinline__ void stash_first(const uint4* sv4, uint4* stash, int ct, int h,
                                            const uint32_t (&vm)[kGroupVecs], float gmax, int jbase, int sg,
                                            GroupCand& cand) {
  int kf = kGroupVecs - 1;
#pragma unroll
  for (int k = kGroupVecs - 2; k >= 0; --k)
    if (vec_max_of<ES>(vm[k]) == gmax) kf = k;
  kf += h * kGroupVecs;
  stash[ct] = sv4[ct + kf * kK1ConsumerThreads];
  cand.stage = sg;
  cand.vec = kf;
  cand.jbase = jbase;
}

// Fold one stage (two halves) into (m, s). s is the sum of 2^(x c - mc) over
// the elements folded so far; mc = m c once m is finite, and before that the
// reference the piece started with (the previous piece's maximum, so the
// first stage needs no second pass in the common case). The exponentials use
// mc from before the stage, so they do not wait on the stage's own maximum.
// When the maximum rises, the sum is moved to the new reference once; the
// halves are re-summed against the new maximum from shared memory only if the
// stage sum overflowed or the new maximum sat more than 2^20 below the old
// reference (where flushed small terms could matter). The argmax keeps the
// vector where the maximum first rose: stages, halves and vectors arrive in
// increasing index order, so a strict '>' (and the lower half and vector on
// a tie) keeps the lowest index.
template <int ES>
__device__ __forceinline__ void fold_stage(const uint4* sv4, uint4* stash, int ct, int jbase, int sg,
                                           float c, float& m, float& mc, float& s, GroupCand& cand) {
  uint32_t w[kGroupWords];
  uint32_t va[kGroupVecs], vb[kGroupVecs];
  load_half(sv4, ct, 0, w);
  const float sa = group_sum<ES>(w, c, mc);
  const float ga = group_max<ES>(w, va);
  load_half(sv4, ct, 1, w);
  const float sb = group_sum<ES>(w, c, mc);
  const float gb = group_max<ES>(w, vb);
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
    const bool lo = ga >= gb;
    uint32_t vm[kGroupVecs];
#pragma unroll
    for (int k = 0; k < kGroupVecs; ++k) vm[k] = lo ? va[k] : vb[k];
    stash_first<ES>(sv4, stash, ct, lo ? 0 : 1, vm, gmax, jbase, sg, cand);
  } else if (gmax > -INFINITY) {
    s += gsum;
  }
}

// Halves of a stage that warp cw folds: a short stage (nvec vectors, the last
// of a piece) holds no data for this warp in half h when the warp's first
// vector of that half, v = 32 cw + 4 h kK1ConsumerThreads, is past nvec; such
// halves are neither masked nor folded. Warp-uniform, so no lane diverges.
__device__ __forceinline__ int stage_halves(int cw, int nvec) {
  if (cw * 32 >= nvec) return 0;
  if (kStageHalves == 1 || cw * 32 + kGroupVecs * kK1ConsumerThreads >= nvec) return 1;
  return 2;
}

// fold_stage over the first `nh` halves of the stage (nh from stage_halves):
// two halves is fold_stage itself; one half folds vectors k = 0..3 only, with
// the same rescaling, re-summing and argmax bookkeeping.
template <int ES>
__device__ __forceinline__ void fold_stage_n(const uint4* sv4, uint4* stash, int ct, int jbase, int sg, float c,
                                             float& m, float& mc, float& s, GroupCand& cand, int nh) {
  if (nh == 2) {
    fold_stage<ES>(sv4, stash, ct, jbase, sg, c, m, mc, s, cand);
    return;
  }
  if (nh == 0) return;
  uint32_t w[kGroupWords];
  uint32_t va[kGroupVecs];
  load_half(sv4, ct, 0, w);
  const float gsum = group_sum<ES>(w, c, mc);
  const float gmax = group_max<ES>(w, va);
  if (gmax > m) {
    const float nmc = gmax * c;
    const float d = mc - nmc;
    if (gsum <= FLT_MAX && d <= 20.f) {
      s = (s + gsum) * ex2(d);
    } else {
      s = (m == -INFINITY ? 0.f : s * ex2(d)) + group_sum<ES>(w, c, nmc);
    }
    m = gmax;
    mc = nmc;
    stash_first<ES>(sv4, stash, ct, 0, va, gmax, jbase, sg, cand);
  } else if (gmax > -INFINITY) {
    s += gsum;
  }
}

// Lowest index in [j0, j1) of the thread's candidate holding the value m,
// read back from its stashed vector; INT_MAX if m is -inf.
template <int ES>
__device__ __forceinline__ int resolve_cand(const GroupCand& cand, const uint4* stash, int ct, float m,
                                            int j0, int j1) {
  if (!(m > -INFINITY)) return INT_MAX;
  if (cand.stage < 0) return cand.j;
  constexpr int N = Elem<ES>::kVec;
  float f[N];
  Elem<ES>::unpack(stash[ct], f);
  const int jv = cand.jbase + (ct + cand.vec * kK1ConsumerThreads) * N;
  int best = INT_MAX;
#pragma unroll
  for (int e = N - 1; e >= 0; --e)
    if (f[e] == m && jv + e >= j0 && jv + e < j1) best = jv + e;
  return best;
}

template <int ES>
__global__ void __maxnreg__(kK1MaxRegs) row_stats_kernel(const RowStatsArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kK1Stages];
  __shared__ __align__(8) uint64_t empty_bar[kK1Stages];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;
  const int64_t E0 = a.T * g / a.G;
  const int64_t E1 = a.T * (g + 1) / a.G;
  const int row0 = static_cast<int>(E0 / a.V);   // the one division; pieces then step row by row
  const int j00 = static_cast<int>(E0 - static_cast<int64_t>(row0) * a.V);

  // Shared-memory setup overlaps the previous kernel's tail, and so does an
  // L2 prefetch of the bytes of the CTA's first kK1Stages copies: a prefetch
  // returns nothing to the program and L2 is where the previous kernel's
  // writes land, so it may run before the dependency wait; the copies after
  // the wait then find those bytes in L2 instead of waiting on DRAM.
  if (tid == 0) {
    for (int i = 0; i < kK1Stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kK1Consumers);
    }
    fence_barrier_init();
    int st = 0;
    for (int row = row0, j0 = j00; E0 < E1 && st < kK1Stages; ++row, j0 = 0) {
      const Piece p = make_piece<ES>(a, row, j0, E1);
      for (int s = 0; s < p.nst && st < kK1Stages; ++s, ++st) {
        const uint32_t off = static_cast<uint32_t>(s) * kK1StageBytes;
        bulk_prefetch_l2(reinterpret_cast<const void*>(p.cp_lo + off),
                         min(static_cast<uint32_t>(kK1StageBytes), static_cast<uint32_t>(p.cp_hi - p.cp_lo) - off));
      }
      if (static_cast<int64_t>(row) * a.V + p.j1 >= E1) break;
    }
  }
  __syncthreads();

  // Inputs may come from the kernel before this one, and the partials this
  // kernel writes may still be read by the previous call: wait for it first.
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0, slot = 0;
      uint32_t phase = 0;   // parity of the current use of `slot`
      bool ok = true;
      for (int row = row0, j0 = j00; E0 < E1 && ok; ++row, j0 = 0) {
        const Piece p = make_piece<ES>(a, row, j0, E1);
        for (int s = 0; s < p.nst; ++s, ++st) {
          // the slot's previous use (parity phase ^ 1) must have been released
          if (st >= kK1Stages && !mbar_wait_bounded(smem_u32(&empty_bar[slot]), phase ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t off = static_cast<uint32_t>(s) * kK1StageBytes;
          const uint32_t bytes = min(static_cast<uint32_t>(kK1StageBytes),
                                     static_cast<uint32_t>(p.cp_hi - p.cp_lo) - off);
          const uint32_t fb = smem_u32(&full_bar[slot]);
          mbar_arrive_expect_tx(fb, bytes);
          bulk_g2s(smem_u32(ring + slot * kK1StageBytes), reinterpret_cast<const void*>(p.cp_lo + off), bytes, fb);
          if (++slot == kK1Stages) {
            slot = 0;
            phase ^= 1;
          }
        }
        if (static_cast<int64_t>(row) * a.V + p.j1 >= E1) break;
      }
      // The copies still in flight are the last (up to) kK1Stages issued; let
      // them land before the CTA can exit.
      for (int k = max(0, st - kK1Stages); k < st; ++k)
        (void)mbar_wait_bounded(smem_u32(&full_bar[k % kK1Stages]), (k / kK1Stages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  uint4* const stash = reinterpret_cast<uint4*>(ring + kK1RingBytes);
  const int ct = tid - 32;
  const int cw = warp - 1;
  const float c = a.c;
  int slot = 0;
  uint32_t phase = 0;
  bool ok = true;
  float ref = 0.f;   // exponent reference a piece starts from (log2 domain)
  for (int row = row0, j0 = j00; E0 < E1; ++row, j0 = 0) {
    const Piece p = make_piece<ES>(a, row, j0, E1);
    float m = -INFINITY, mc = ref, s = 0.f;
    GroupCand cand;
    cand.stage = -1;
    cand.vec = 0;
    cand.j = INT_MAX;
    cand.jbase = 0;
    for (int j = p.j0 + ct; j < p.head_end; j += kK1ConsumerThreads)
      fold_scalar(Elem<ES>::load(p.rowp, j), j, c, m, mc, s, cand);
    // Per-piece constants; the stage loop only steps them.
    const int last = p.nst - 1;
    const bool first_edge = p.cp_lo < p.lo;
    const bool last_hull = p.cp_hi > p.hi;
    const int last_nvec =
        static_cast<int>((p.cp_hi - p.cp_lo - static_cast<uintptr_t>(last > 0 ? last : 0) * kK1StageBytes) / 16u);
    const bool last_edge = last_hull || last_nvec != kStageFullVecs;
    // row index of the piece's first copied element (may precede j0 by up to 7)
    const int jbase0 = p.j0 - static_cast<int>((p.lo - p.cp_lo) / ES);
    int jbase = jbase0;
    for (int sg = 0; sg < p.nst; ++sg) {
      if (ok) {
        if (!mbar_wait_bounded(smem_u32(&full_bar[slot]), phase)) {
          ok = false;   // stop consuming (and releasing); the producer times out too
        } else {
          uint4* sv4 = reinterpret_cast<uint4*>(ring + slot * kK1StageBytes);
          const int nh = sg == last ? stage_halves(cw, last_nvec) : kStageHalves;
          if ((sg == 0 && first_edge) || (sg == last && last_edge)) {
            const int nvec = sg == last ? last_nvec : kStageFullVecs;
            mask_stage<ES>(sv4, ct, nvec, jbase, p.j0, p.j1, (sg == 0 && first_edge) ? 0 : -1,
                           (sg == last && last_hull) ? nvec - 1 : -1, nh);
          }
          fold_stage_n<ES>(sv4, stash, ct, jbase, sg, c, m, mc, s, cand, nh);
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
        }
      }
      jbase += kK1StageBytes / ES;
      if (++slot == kK1Stages) {
        slot = 0;
        phase ^= 1;
      }
    }
    for (int j = p.tail_begin + ct; j < p.j1; j += kK1ConsumerThreads)
      fold_scalar(Elem<ES>::load(p.rowp, j), j, c, m, mc, s, cand);
    if (m > -INFINITY) ref = mc;

    // Warp: max, the lowest index among lanes holding it, and the sum
    // rescaled to the warp max (fixed shuffle order).
    const float wm = warp_max(m);
    const int widx = warp_min_nonneg((m == wm) ? resolve_cand<ES>(cand, stash, ct, m, p.j0, p.j1) : INT_MAX);
    float ws = (m == -INFINITY) ? 0.f : s * ex2((m - wm) * c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);

    // One partial per warp and piece, at slot (row + g) * kK1Consumers + cw:
    // the decide kernel merges a row's partials, so no warp waits for,
    // counts or merges another warp's result here.
    if (lane == 0) {
      Partial out;
      out.m = wm;
      out.s = ws;
      out.idx = widx;
      out.err = ok ? 0 : 1;
      store_partial_keep(a.partials + (static_cast<int64_t>(p.row) + g) * kK1Consumers + cw, out);
    }
    if (static_cast<int64_t>(row) * a.V + p.j1 >= E1) break;
  }
}

// One row's partials: kK1Consumers per CTA whose range meets the row, at
// slots (row + g) * kK1Consumers + w, contiguous for one CTA. A CTA's
// partials are folded as a pairwise tree, and the CTAs in increasing order;
// the order is fixed, so the result is deterministic.
__device__ __forceinline__ void load_cta_partials(const Partial* __restrict__ parts, int64_t row, int g,
                                                  Partial (&v)[kK1Consumers]) {
  const Partial* p = parts + (row + g) * kK1Consumers;
#pragma unroll
  for (int w = 0; w < kK1Consumers; ++w) v[w] = p[w];
}

// Pairwise merge of one CTA's warp partials (w, w + 1), (w, w + 2), ...
__device__ __forceinline__ void merge_cta_partials(const Partial (&v)[kK1Consumers], float c, float& m, float& s,
                                                   int& idx, int& err) {
  float tm[kK1Consumers], ts[kK1Consumers];
  int ti[kK1Consumers];
  err = 0;
#pragma unroll
  for (int w = 0; w < kK1Consumers; ++w) {
    tm[w] = v[w].m;
    ts[w] = v[w].s;
    ti[w] = v[w].idx;
    err |= v[w].err;
  }
#pragma unroll
  for (int step = 1; step < kK1Consumers; step <<= 1)
#pragma unroll
    for (int w = 0; w + step < kK1Consumers; w += 2 * step) merge_stats(tm[w], ts[w], ti[w], tm[w + step], ts[w + step], ti[w + step], c);
  m = tm[0];
  s = ts[0];
  idx = ti[0];
}

// Block-cooperative staging. The slots (row + g) of consecutive rows are
// consecutive (a CTA's range continues into the next row), so rows
// [r0, r1] own the dense slot range [r0 + g_lo(r0), r1 + g_hi(r1)]. Each
// thread of the block merges the kK1Consumers warp partials of one slot into
// one Partial in shared memory; a row's thread then merges its few slots with
// merge_row_staged. Same merge order as merge_row_serial, so the results
// are identical.
struct SlotRange {
  int64_t lo;   // first slot
  int n;        // slots
};

__device__ __forceinline__ SlotRange slot_range(int64_t r0, int64_t r1, int V, int64_t T, int G) {
  SlotRange sr;
  sr.lo = r0 + cta_of(r0 * V, T, G);
  const int64_t hi = r1 + cta_of(r1 * V + V - 1, T, G);
  sr.n = static_cast<int>(hi - sr.lo + 1);
  return sr;
}

// Stages two slot ranges in one pass (a second range of n = 0 is skipped), so
// the loads of both are in flight together.
__device__ __forceinline__ void stage_slots(const Partial* __restrict__ parts, const SlotRange& sa, Partial* staged_a,
                                            const SlotRange& sb, Partial* staged_b, float c) {
  const int n = sa.n + sb.n;
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    const bool first = q < sa.n;
    const int k = first ? q : q - sa.n;
    Partial v[kK1Consumers];
    const Partial* p = parts + ((first ? sa.lo : sb.lo) + k) * kK1Consumers;
#pragma unroll
    for (int w = 0; w < kK1Consumers; ++w) v[w] = p[w];
    Partial o;
    merge_cta_partials(v, c, o.m, o.s, o.idx, o.err);
    (first ? staged_a : staged_b)[k] = o;
  }
}

__device__ __forceinline__ void merge_row_staged(const Partial* staged, const SlotRange& sr, int64_t row, int V,
                                                 int64_t T, int G, float c, float& m, float& s, int& idx, int& err) {
  const int64_t e0 = row * V;
  const int q0 = static_cast<int>(row + cta_of(e0, T, G) - sr.lo);
  const int q1 = static_cast<int>(row + cta_of(e0 + V - 1, T, G) - sr.lo);
  m = -INFINITY;
  s = 0.f;
  idx = INT_MAX;
  err = 0;
  for (int q = q0; q <= q1; ++q) {
    const Partial v = staged[q];
    merge_stats(m, s, idx, v.m, v.s, v.idx, c);
    err |= v.err;
  }
  if (m == -INFINITY) idx = 0;   // every element is -inf: the lowest index attains the max
}

// One row's statistics merged by a half-warp (lane16 = lane & 15): lane l
// takes partials l, l + 16, ... of the row's (g_hi - g_lo + 1) * kK1Consumers
// (in slot order), merges them, and four xor-shuffle levels within the half
// merge the lanes, so every lane of the half ends with the row's statistics.
// All 32 lanes of the warp must call it (valid = false: a half with no row,
// which contributes nothing); merge_stats is symmetric, so both partners of a
// shuffle compute the same value and the result is deterministic. LOADS
// partials per lane are loaded before any of them is merged (one L2 round
// trip for rows of up to 16 LOADS partials); a lane merges its partials in
// increasing k whatever LOADS is, so the result does not depend on it.
template <int LOADS = 2>
__device__ __forceinline__ void merge_row_half(const Partial* __restrict__ parts, int64_t row, bool valid, int V,
                                               int64_t T, int G, float c, int lane16, float& m, float& s, int& idx,
                                               int& err) {
  m = -INFINITY;
  s = 0.f;
  idx = INT_MAX;
  err = 0;
  if (valid) {
    const int64_t e0 = row * V;
    const int g_lo = cta_of(e0, T, G), g_hi = cta_of(e0 + V - 1, T, G);
    const int n = (g_hi - g_lo + 1) * kK1Consumers;
    const Partial* p = parts + (row + g_lo) * kK1Consumers;
    if constexpr (LOADS == 2) {
      for (int k = lane16; k < n; k += 32) {
        const Partial v0 = p[k];
        Partial v1;
        if (k + 16 < n) v1 = p[k + 16];
        merge_stats(m, s, idx, v0.m, v0.s, v0.idx, c);
        err |= v0.err;
        if (k + 16 < n) {
          merge_stats(m, s, idx, v1.m, v1.s, v1.idx, c);
          err |= v1.err;
        }
      }
    } else {
      for (int k0 = lane16; k0 < n; k0 += 16 * LOADS) {
        Partial v[LOADS];
#pragma unroll
        for (int u = 0; u < LOADS; ++u)
          if (k0 + 16 * u < n) v[u] = p[k0 + 16 * u];
#pragma unroll
        for (int u = 0; u < LOADS; ++u) {
          if (k0 + 16 * u < n) {
            merge_stats(m, s, idx, v[u].m, v[u].s, v[u].idx, c);
            err |= v[u].err;
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    err |= __shfl_xor_sync(0xffffffffu, err, o);
    merge_stats(m, s, idx, om, os, oi, c);
  }
  if (m == -INFINITY) idx = 0;   // every element is -inf: the lowest index attains the max
}

// Merge one row's partials CTA by CTA (few registers). The decide kernels
// use it when a block's slots exceed their staging area; the mu pass always.
__device__ __noinline__ void merge_row_serial(const Partial* __restrict__ parts, int64_t row, int V, int64_t T,
                                              int G, float c, float& m, float& s, int& idx, int& err) {
  const int64_t e0 = row * V;
  const int g_lo = cta_of(e0, T, G), g_hi = cta_of(e0 + V - 1, T, G);
  m = -INFINITY;
  s = 0.f;
  idx = INT_MAX;
  err = 0;
  for (int g = g_lo; g <= g_hi; ++g) {
    Partial v[kK1Consumers];
    load_cta_partials(parts, row, g, v);
    float cm, cs;
    int ci, ce;
    merge_cta_partials(v, c, cm, cs, ci, ce);
    merge_stats(m, s, idx, cm, cs, ci, c);
    err |= ce;
  }
  if (m == -INFINITY) idx = 0;   // every element is -inf: the lowest index attains the max
}


}  // namespace sv
