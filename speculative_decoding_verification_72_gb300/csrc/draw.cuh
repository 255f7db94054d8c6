// K3: the one draw per request that ends a stochastic round (spec-decode
// README, "How it works": on the first rejection a sample from
// normalize(relu(p - q)); after K acceptances a bonus sample from p; the
// nanospec README's tree and deterministic-draft rules draw from p with the
// rejected tokens removed).
//
// The draw is an inverse CDF over the row's weights w_j in index order. It
// runs as two kernels:
//
//  * draw_sum_kernel (K3a) streams the drawn rows once and writes, per
//    request b and vocabulary chunk k (kK3ChunkBytes of each row), the pair
//    (sum w, sum p) over the chunk. It is persistent and warp-specialized like
//    the row-statistics pass: the B * P (request, chunk) items are split into
//    equal contiguous ranges, one per CTA; warp 0's lane 0 copies each item's
//    target chunk (and draft chunk for a residual) into a 6-stage
//    shared-memory ring with 1-D bulk copies (TMA), and 7 consumer warps sum
//    the weights from shared memory. The last consumer warp to finish an item
//    merges the warps' sums in a fixed order and writes them, so no warp waits
//    for another. Copies cover the 16-byte-aligned hull of a chunk (clipped to
//    the caller's buffer); elements outside the chunk are skipped and the few
//    elements a clipped hull misses are read from global memory.
//  * draw_pick_kernel (K3b), one CTA per request, forms the ordered prefix of
//    the chunk sums with fp32 warp scans, finds the chunk where u * S falls,
//    loads that chunk (one 16-byte vector per thread and row, so each thread
//    owns a contiguous run of elements), and resolves the smallest j whose
//    inclusive prefix sum exceeds u * S with a block scan. The drawn token's
//    logit stays in the picking thread's registers for the log-prob and mu.
//
// Per-element weights come from weight_of in both kernels. A wait that gives
// up marks every chunk sum of the CTA's range NaN; the pick kernel then
// reports status bit 32 for that request.
#pragma once

#include "finish.cuh"
#include "row_stats.cuh"
#include "sv_common.cuh"

namespace sv {

constexpr int kK3Consumers = 7;
constexpr int kK3Threads = 32 * (kK3Consumers + 1);
constexpr int kK3ConsumerThreads = 32 * kK3Consumers;
constexpr int kK3CtasPerSm = 2;
constexpr int kK3ChunkBytes = 16384;                   // per row and chunk
constexpr int kK3SlotBytes = kK3ChunkBytes + 32;      // a chunk's 16-byte hull
constexpr int kK3Stages = 6;
constexpr int kK3SmemBytes = kK3Stages * kK3SlotBytes;
constexpr int kK3Req = 8;           // requests whose descriptor and exclusions a CTA caches
constexpr int kK3LocalExcl = 64;    // exclusions cached per request
constexpr int kK3MaxChunks = 256;   // chunk sums the pick kernel stages in shared memory
constexpr int kK3PickThreads = 1024;
constexpr int kStatusWaitErr = SV_STATUS_TIMEOUT;
// Fused decision: chains of at most kFusedMaxRows positions (K + 1).
constexpr int kFusedMaxRows = 16;
constexpr int kFusedRowsPerReq = 2 * kFusedMaxRows - 1;   // target rows 0..K, draft rows 0..K-1

template <int ES>
constexpr int kK3ChunkElems = kK3ChunkBytes / ES;
// Elements one pick thread owns in the chosen chunk: one 16-byte vector.
template <int ES>
constexpr int kK3PickElems = kK3ChunkElems<ES> / kK3PickThreads;

struct DrawArgs {
  const uint8_t* tgt;
  int64_t tgt_stride;   // bytes
  uintptr_t tgt_lo, tgt_hi;   // bytes the target buffer holds
  const uint8_t* dft;
  int64_t dft_stride;   // bytes
  uintptr_t dft_lo, dft_hi;
  int32_t V, P, chunk_elems;
  int32_t B;
  int32_t G;            // K3a CTAs
  float c;              // log2(e) / T
  const DrawDesc* draws;
  const int32_t* excl;
  int32_t excl_stride;
  float2* part;         // [B * P]: (sum w, sum p)
  int32_t out_cols;
  int32_t* out_tokens;
  float* out_logprob;
  float* out_mu;
  int32_t* out_nodes;    // tree calls, else nullptr
  int32_t* out_status;
  FinishArgs fin;        // applied by the pick kernel when fin_here
  int32_t fin_here;
  // Fused decision (stochastic chain, draft logits, exact rule, K + 1 <=
  // kFusedMaxRows): draw_sum_kernel decides its own requests from the row
  // pass's partials (the same half-warp merges and acceptance tests as the
  // decide kernel) instead of reading a decide kernel's descriptors. The CTA
  // whose range holds a request's first chunk writes that request's
  // accepted outputs, count, status and draw descriptor (for the pick).
  int32_t fused;
  const Partial* k1_part;
  int64_t k1_T;
  int32_t k1_G;
  int32_t K;
  const int32_t* drafts;     // [B, K]
  const float* uniforms;     // [B, K + 1]
  int32_t* out_num;          // [B]
  DrawDesc* draws_out;       // [B]: the same array as draws
};

// Weights of one element from its logits: p = 2^(x c - lp2), w = relu(p - q)
// for a residual, else p.
__device__ __forceinline__ void weight_of(float x, float y, bool resid, float c, float lp2, float lq2,
                                          float& w, float& p) {
  p = ex2(fmaf(x, c, -lp2));
  w = resid ? fmaxf(p - ex2(fmaf(y, c, -lq2)), 0.f) : p;
}

// ------------------------------------------------------------------ K3a

// One copied row chunk, as the producer describes it to the consumers. A
// masked draw's excluded tokens that fall in the chunk travel with it (the
// first kStageExcl; with more, consumers scan the request's whole list).
constexpr int kStageExcl = 4;
struct StageDesc {
  const uint8_t* rowp;   // row start
  const int32_t* xl;     // the request's exclusion list (shared or global memory)
  int32_t item;          // b * P + k; -1 ends the stream
  int32_t e0;            // row index of the copy's first element (may precede the chunk)
  int32_t nel;           // elements copied (0: nothing copied)
  int32_t type;          // DrawType
  int32_t nx;            // excluded tokens inside the chunk
  int32_t nxl;           // length of xl
  float lp2, lq2;
  int32_t x[kStageExcl];
};

// A descriptor read with volatile loads: only requests past the CTA's cache
// take this path, and the compiler may not hoist it onto the common one (a
// speculated global load there cost the producer a round trip per item).
__device__ __forceinline__ uint4 ld_volatile_v4(const void* p) {
  uint4 q;
  asm volatile("ld.volatile.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
               : "l"(p));
  return q;
}

__device__ __forceinline__ DrawDesc load_desc_volatile(const DrawDesc* p) {
  static_assert(sizeof(DrawDesc) == 48, "three 16-byte words");
  const uint4 q0 = ld_volatile_v4(p);
  const uint4 q1 = ld_volatile_v4(reinterpret_cast<const uint4*>(p) + 1);
  const uint4 q2 = ld_volatile_v4(reinterpret_cast<const uint4*>(p) + 2);
  DrawDesc d;
  d.type = static_cast<int32_t>(q0.x);
  d.t_row = static_cast<int32_t>(q0.y);
  d.d_row = static_cast<int32_t>(q0.z);
  d.pos = static_cast<int32_t>(q0.w);
  d.u = __uint_as_float(q1.x);
  d.lp2 = __uint_as_float(q1.y);
  d.lq2 = __uint_as_float(q1.z);
  d.scale = __uint_as_float(q1.w);
  d.n_excl = static_cast<int32_t>(q2.x);
  d.pad0 = static_cast<int32_t>(q2.y);
  d.pad1 = static_cast<int32_t>(q2.z);
  d.pad2 = static_cast<int32_t>(q2.w);
  return d;
}

// 16-byte-aligned hull of elements [lo, hi) of a row, clipped to [safe_lo, safe_hi).
template <int ES>
__device__ __forceinline__ void chunk_hull(const uint8_t* rowp, int lo, int hi, uintptr_t safe_lo,
                                           uintptr_t safe_hi, uintptr_t& clo, uint32_t& bytes, int& e0) {
  const uintptr_t L = reinterpret_cast<uintptr_t>(rowp) + static_cast<uintptr_t>(lo) * ES;
  const uintptr_t H = reinterpret_cast<uintptr_t>(rowp) + static_cast<uintptr_t>(hi) * ES;
  uintptr_t a = L & ~static_cast<uintptr_t>(15);
  if (a < safe_lo) a = (L + 15) & ~static_cast<uintptr_t>(15);
  uintptr_t z = (H + 15) & ~static_cast<uintptr_t>(15);
  if (z > safe_hi) z = H & ~static_cast<uintptr_t>(15);
  if (z <= a) {
    clo = 0;
    bytes = 0;
    e0 = lo;
    return;
  }
  clo = a;
  bytes = static_cast<uint32_t>(z - a);
  e0 = static_cast<int>((static_cast<int64_t>(a) - static_cast<int64_t>(reinterpret_cast<uintptr_t>(rowp))) / ES);
}

// Element j of a row from its stage copy when the copy holds it, else from
// global memory.
template <int ES>
__device__ __forceinline__ float stage_elem(const uint8_t* sm, const StageDesc& s, int j) {
  const int k = j - s.e0;
  if (k >= 0 && k < s.nel) {
    if constexpr (ES == 4) return reinterpret_cast<const float*>(sm)[k];
    else return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short*>(sm)[k]) << 16);
  }
  return Elem<ES>::load(s.rowp, j);
}

// Bit e set when element jv + e (e < n) is on the list.
__device__ __forceinline__ uint32_t excl_bits(int jv, int n, int nex, const int* lst) {
  uint32_t m = 0u;
  for (int r = 0; r < nex; ++r) {
    const unsigned d = static_cast<unsigned>(lst[r] - jv);
    if (d < static_cast<unsigned>(n)) m |= 1u << d;
  }
  return m;
}

__device__ __forceinline__ bool stage_excludes(const StageDesc& s, int j) {
  if (s.nx <= kStageExcl) {
    bool hit = false;
#pragma unroll
    for (int r = 0; r < kStageExcl; ++r) hit |= (r < s.nx && s.x[r] == j);
    return hit;
  }
  return excl_bits(j, 1, s.nxl, s.xl) != 0u;
}

// A pair of elements as two floats (bf16: one 32-bit word; fp32: two).
template <int ES>
__device__ __forceinline__ float2 pair_of(const uint4& q, int i) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  if constexpr (ES == 2) return make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  else return make_float2(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}

// The (sum w, sum p) share of consumer thread ct over one copied chunk
// [lo, hi). Vectors wholly inside the chunk and free of excluded tokens take
// the packed fp32x2 path (the same per-element arithmetic as weight_of, two
// lanes at a time); the chunk's edge vectors and those holding an excluded
// token go element by element.
template <int ES, bool RESID>
__device__ __forceinline__ void sum_stage(const StageDesc& ts, const StageDesc& ds, const uint8_t* tsm,
                                          const uint8_t* dsm, int lo, int hi, int ct, float c, float& sw,
                                          float& sp) {
  constexpr int N = Elem<ES>::kVec;
  const uint4* tv = reinterpret_cast<const uint4*>(tsm);
  const uint4* dv = reinterpret_cast<const uint4*>(dsm);
  const float2 c2 = make_float2(c, c);
  const float2 nlp = make_float2(-ts.lp2, -ts.lp2);
  const float2 nlq = make_float2(-ts.lq2, -ts.lq2);
  float2 accp[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float2 accw[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float sws = 0.f, sps = 0.f;
  if (!RESID || (ds.e0 == ts.e0 && ds.nel == ts.nel)) {
    // (for a residual the draft copy holds the same elements at the same places)
    const int nv = ts.nel / N;
    const int dlo = lo - ts.e0, dhi = hi - ts.e0;
    const int v_lo = dlo <= 0 ? 0 : (dlo + N - 1) / N;
    const int v_hi = min(nv, dhi / N);
    const bool all_slow = ts.nx > kStageExcl;
    uint32_t xmask = 0u;   // bit i: this thread's i-th vector holds an excluded token
    if (!all_slow) {
#pragma unroll
      for (int r = 0; r < kStageExcl; ++r) {
        const int d = ts.x[r] - ts.e0;
        if (r < ts.nx && d >= 0) {
          const int vt = d / N;
          if (vt < nv && vt % kK3ConsumerThreads == ct) xmask |= 1u << (vt / kK3ConsumerThreads);
        }
      }
    }
    int i = 0;
    for (int v = ct; v < nv; v += kK3ConsumerThreads, ++i) {
      if (!all_slow && v >= v_lo && v < v_hi && !((xmask >> i) & 1u)) {
        const uint4 xq = tv[v];
        uint4 yq;
        if (RESID) yq = dv[v];
#pragma unroll
        for (int h = 0; h < N / 2; ++h) {
          const float2 t = __ffma2_rn(pair_of<ES>(xq, h), c2, nlp);
          const float2 pp = make_float2(ex2(t.x), ex2(t.y));
          accp[h & 1] = __fadd2_rn(accp[h & 1], pp);
          if (RESID) {
            const float2 u = __ffma2_rn(pair_of<ES>(yq, h), c2, nlq);
            const float2 w = make_float2(fmaxf(pp.x - ex2(u.x), 0.f), fmaxf(pp.y - ex2(u.y), 0.f));
            accw[h & 1] = __fadd2_rn(accw[h & 1], w);
          }
        }
      } else {
        const int jv = ts.e0 + v * N;
        float xf[N], yf[N];
        Elem<ES>::unpack(tv[v], xf);
        if (RESID) Elem<ES>::unpack(dv[v], yf);
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const int j = jv + e;
          if (j >= lo && j < hi) {
            float w, p;
            weight_of(xf[e], RESID ? yf[e] : 0.f, RESID, c, ts.lp2, ts.lq2, w, p);
            if (!RESID && ts.nx && stage_excludes(ts, j)) w = 0.f;
            sws += w;
            sps += p;
          }
        }
      }
    }
    // Elements of the chunk the (clipped) copy does not hold, from global memory.
    const int c_lo = ts.nel ? max(lo, ts.e0) : hi;
    const int c_hi = ts.nel ? min(hi, ts.e0 + ts.nel) : hi;
    int j = -1;
    if (ct < c_lo - lo) j = lo + ct;
    else if (ct - (c_lo - lo) < hi - c_hi) j = c_hi + ct - (c_lo - lo);
    if (j >= 0 && j < hi && (j < c_lo || j >= c_hi)) {
      float w, p;
      const float x = Elem<ES>::load(ts.rowp, j);
      const float y = RESID ? Elem<ES>::load(ds.rowp, j) : 0.f;
      weight_of(x, y, RESID, c, ts.lp2, ts.lq2, w, p);
      if (!RESID && ts.nx && stage_excludes(ts, j)) w = 0.f;
      sws += w;
      sps += p;
    }
  } else {
    // Target and draft copies hold different element ranges: element by element.
    for (int j = lo + ct; j < hi; j += kK3ConsumerThreads) {
      float w, p;
      weight_of(stage_elem<ES>(tsm, ts, j), stage_elem<ES>(dsm, ds, j), true, c, ts.lp2, ts.lq2, w, p);
      sws += w;
      sps += p;
    }
  }
  const float2 ap = __fadd2_rn(accp[0], accp[1]);
  sp = (ap.x + ap.y) + sps;
  if (RESID) {
    const float2 aw = __fadd2_rn(accw[0], accw[1]);
    sw = (aw.x + aw.y) + sws;
  } else {
    sw = (ap.x + ap.y) + sws;   // w = p away from excluded tokens
  }
}

// Fused decision for the requests b_first .. b_first + nreq - 1 of a draw-sum
// CTA (stochastic chain, draft logits, exact rule; spec-decode README, "How
// it works"): accept draft i with probability min(1, p(d_i)/q(d_i)), stop at
// the first rejection n (residual draw from normalize(relu(p - q)) at row n),
// else a bonus draw from p at row K. The same arithmetic, merge order and
// status bits as the decide kernel's stochastic path, so the outputs are
// identical. Block-cooperative: every thread calls it.
template <int ES>
__device__ __forceinline__ void fused_decide(const DrawArgs& a, int b_first, int nreq, int64_t i0, int64_t i1,
                                             int tok, bool bad, float x, float y, float u, float uK, Partial* s_rs,
                                             DrawDesc* s_desc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = a.K, R = K + 1, per = 2 * K + 1;
  const float c = a.c;
  // Row statistics, one half-warp per row (the decide kernel's merge).
  const int rows_all = nreq * per;
  for (int q0 = 0; q0 < rows_all; q0 += kK3Threads / 16) {
    const int q = q0 + (tid >> 4);
    const bool valid = q < rows_all;
    const int r = valid ? q / per : 0, j = valid ? q - r * per : 0;
    const int64_t bq = b_first + r;
    const int64_t row = j <= K ? bq * R + j : static_cast<int64_t>(a.B) * R + bq * K + (j - K - 1);
    float m, s;
    int idx, err;
    merge_row_half(a.k1_part, row, valid, a.V, a.k1_T, a.k1_G, c, tid & 15, m, s, idx, err);
    if (valid && (tid & 15) == 0) {
      Partial o;
      o.m = m;
      o.s = s;
      o.idx = idx;
      o.err = err;
      s_rs[q] = o;
    }
  }
  __syncthreads();
  if (warp >= nreq) return;
  const int b = b_first + warp;
  const Partial tr = s_rs[warp * per + min(lane, K)];
  const float lp2row = tr.m * c + log2f(tr.s);
  int st = 0;
  if (!(fabsf(tr.m) <= FLT_MAX) || !(tr.s > 0.f && tr.s <= FLT_MAX)) st |= SV_STATUS_NONFINITE_ROW;
  if (tr.err) st |= SV_STATUS_TIMEOUT;
  float lq2row = 0.f, lp2 = 0.f, acc = 0.f;
  bool zero = false, rej = false;
  if (lane < K) {
    const Partial dr = s_rs[warp * per + K + 1 + lane];
    lq2row = dr.m * c + log2f(dr.s);
    if (!(fabsf(dr.m) <= FLT_MAX) || !(dr.s > 0.f && dr.s <= FLT_MAX)) st |= SV_STATUS_NONFINITE_ROW;
    if (dr.err) st |= SV_STATUS_TIMEOUT;
    if (!bad) {
      lp2 = x * c - lp2row;   // log2 p(t)
      const float lq2 = y * c - lq2row;
      if (lp2 == -INFINITY && lq2 == -INFINITY) zero = true;
      else acc = ex2(fminf(0.f, lp2 - lq2));   // min(1, p/q)
    }
    rej = bad || zero || !(u < acc);
  }
  const unsigned rm = __ballot_sync(0xffffffffu, lane < K && rej);
  const int n = rm ? __ffs(rm) - 1 : K;
  int stat = lane <= n ? st : 0;
  if (lane == n && n < K) {
    if (bad) stat |= SV_STATUS_BAD_TOKEN;
    if (zero) stat |= SV_STATUS_ZERO_MASS;
  }
  stat = __reduce_or_sync(0xffffffffu, stat);
  DrawDesc d;
  d.type = n == K ? kDrawP : kDrawResid;
  d.t_row = b * R + n;
  d.d_row = b * K + n;
  d.pos = n;
  d.u = uK;
  d.lp2 = __shfl_sync(0xffffffffu, lp2row, n);
  d.lq2 = n < K ? __shfl_sync(0xffffffffu, lq2row, n) : 0.f;
  d.scale = 1.f;
  d.n_excl = 0;
  d.pad0 = d.pad1 = d.pad2 = 0;
  if (lane == 0) s_desc[warp] = d;
  // The CTA holding the request's first chunk writes its outputs once.
  const int64_t first_item = static_cast<int64_t>(b) * a.P;
  if (first_item >= i0 && first_item < i1) {
    if (lane == 0) {
      a.draws_out[b] = d;
      a.out_num[b] = n;
      if (a.out_status) a.out_status[b] = stat;
    }
    if (lane < R && lane != n) {   // the pick kernel writes position n
      const int64_t o = static_cast<int64_t>(b) * a.out_cols + lane;
      a.out_tokens[o] = lane < n ? tok : -1;
      if (a.out_logprob) a.out_logprob[o] = lane < n ? lp2 * kLn2 : 0.f;
      if (a.out_mu) a.out_mu[o] = lane < n ? ex2(lp2) : 0.f;
    }
  }
}

template <int ES>
__global__ void __launch_bounds__(kK3Threads, kK3CtasPerSm) draw_sum_kernel(const DrawArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kK3Stages];
  __shared__ __align__(8) uint64_t empty_bar[kK3Stages];
  __shared__ StageDesc sdesc[kK3Stages];
  __shared__ float2 red[kK3Stages][kK3Consumers];
  __shared__ int red_cnt[kK3Stages];
  __shared__ DrawDesc s_desc[kK3Req];
  __shared__ int s_ex[kK3Req][kK3LocalExcl];
  __shared__ int s_err;
  __shared__ Partial s_rs[kK3Req * kFusedRowsPerReq];   // fused decision: row statistics

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t n_items = static_cast<int64_t>(a.B) * a.P;
  const int64_t i0 = n_items * blockIdx.x / a.G;
  const int64_t i1 = n_items * (blockIdx.x + 1) / a.G;
  const int b_first = static_cast<int>(i0 / a.P);

  // Fused decision: warp w decides request b_first + w, lane i position i.
  // Its call inputs (draft tokens, uniforms, the draft tokens' logits) are
  // read before the dependency wait.
  const int R = a.K + 1;
  const int nreq_f = a.fused ? min(kK3Req, static_cast<int>((i1 - 1) / a.P) - b_first + 1) : 0;
  int f_tok = -1;
  bool f_bad = false;
  float f_x = -INFINITY, f_y = -INFINITY, f_u = 0.f, f_uK = 0.f;
  if (warp < nreq_f) {
    const int64_t bq = b_first + warp;
    f_uK = a.uniforms[bq * R + a.K];
    if (lane < a.K) {
      f_tok = a.drafts[bq * a.K + lane];
      f_bad = f_tok < 0 || f_tok >= a.V;
      f_u = a.uniforms[bq * R + lane];
      if (!f_bad) {
        f_x = Elem<ES>::load(a.tgt + (bq * R + lane) * a.tgt_stride, f_tok);
        f_y = Elem<ES>::load(a.dft + (bq * a.K + lane) * a.dft_stride, f_tok);
      }
    }
  }

  // Shared-memory setup overlaps the decide kernel's tail.
  if (tid < kK3Stages) red_cnt[tid] = 0;
  if (tid == 0) {
    s_err = 0;
    for (int i = 0; i < kK3Stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kK3Consumers);
    }
    fence_barrier_init();
  }
  grid_dep_wait();   // the draw descriptors come from the decide kernel (or the row pass, fused)
  grid_dep_launch();

  if (a.fused) {
    fused_decide<ES>(a, b_first, nreq_f, i0, i1, f_tok, f_bad, f_x, f_y, f_u, f_uK, s_rs, s_desc);
  } else {
    // Descriptors and exclusion lists of the first kK3Req requests of the range.
    const int nreq = min(kK3Req, static_cast<int>((i1 - 1) / a.P) - b_first + 1);
    if (tid < nreq) s_desc[tid] = a.draws[b_first + tid];
    for (int x = tid; x < nreq * kK3LocalExcl; x += kK3Threads) {
      const int r = x / kK3LocalExcl, e = x - r * kK3LocalExcl;
      if (e < a.excl_stride) s_ex[r][e] = a.excl[static_cast<int64_t>(b_first + r) * a.excl_stride + e];
    }
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0, slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      int b = b_first, k = static_cast<int>(i0 - static_cast<int64_t>(b_first) * a.P);
      // Claim the next slot: its previous use has been released.
      auto claim = [&]() -> bool {
        return st < kK3Stages || mbar_wait_bounded(smem_u32(&empty_bar[slot]), phase ^ 1);
      };
      auto advance = [&]() {
        ++st;
        if (++slot == kK3Stages) {
          slot = 0;
          phase ^= 1;
        }
      };
      for (int64_t i = i0; i < i1 && ok; ++i) {
        const int r = b - b_first;
        const DrawDesc d = r < kK3Req ? s_desc[r] : load_desc_volatile(a.draws + b);
        if (d.type != kDrawNone) {
          const int lo = k * a.chunk_elems;
          const int hi = min(a.V, lo + a.chunk_elems);
          StageDesc sd;
          sd.item = static_cast<int32_t>(i);
          sd.type = d.type;
          sd.lp2 = d.lp2;
          sd.lq2 = d.lq2;
          sd.nx = 0;
          sd.nxl = d.type == kDrawMaskedP ? d.n_excl : 0;
          sd.xl = (r < kK3Req && sd.nxl <= kK3LocalExcl) ? s_ex[r] : a.excl + static_cast<int64_t>(b) * a.excl_stride;
#pragma unroll
          for (int q = 0; q < kStageExcl; ++q) sd.x[q] = -1;
          for (int q = 0; q < sd.nxl; ++q) {
            const int t = sd.xl[q];
            if (t >= lo && t < hi) {
#pragma unroll
              for (int u = 0; u < kStageExcl; ++u)
                if (sd.nx == u) sd.x[u] = t;
              ++sd.nx;
            }
          }
          const int nrow = d.type == kDrawResid ? 2 : 1;
          for (int h = 0; h < nrow && ok; ++h) {
            sd.rowp = h == 0 ? a.tgt + static_cast<int64_t>(d.t_row) * a.tgt_stride
                             : a.dft + static_cast<int64_t>(d.d_row) * a.dft_stride;
            uintptr_t clo;
            uint32_t bytes;
            chunk_hull<ES>(sd.rowp, lo, hi, h == 0 ? a.tgt_lo : a.dft_lo, h == 0 ? a.tgt_hi : a.dft_hi, clo,
                           bytes, sd.e0);
            sd.nel = static_cast<int32_t>(bytes / ES);
            if (!claim()) {
              ok = false;
              break;
            }
            sdesc[slot] = sd;
            const uint32_t fb = smem_u32(&full_bar[slot]);
            mbar_arrive_expect_tx(fb, bytes);
            if (bytes) bulk_g2s(smem_u32(ring + slot * kK3SlotBytes), reinterpret_cast<const void*>(clo), bytes, fb);
            advance();
          }
        }
        if (++k == a.P) {
          k = 0;
          ++b;
        }
      }
      bool ended = false;
      if (ok) {   // end of stream: a descriptor with no copy
        StageDesc sd;
        sd.rowp = nullptr;
        sd.xl = nullptr;
        sd.item = -1;
        sd.e0 = sd.nel = sd.type = sd.nx = sd.nxl = 0;
        sd.lp2 = sd.lq2 = 0.f;
        if (claim()) {
          sdesc[slot] = sd;
          mbar_arrive(smem_u32(&full_bar[slot]));
          ended = true;
        } else {
          ok = false;
        }
      }
      if (!ok) atomicOr(&s_err, 1);
      // Copies still in flight (among the last kK3Stages issued) land before
      // the CTA exits. The end marker reused the slot of stage st - kK3Stages
      // after its release, so that copy has landed (and its parity is taken).
      for (int q = max(0, st - kK3Stages + (ended ? 1 : 0)); q < st; ++q)
        (void)mbar_wait_bounded(smem_u32(&full_bar[q % kK3Stages]), (q / kK3Stages) & 1);
    }
    __syncwarp();   // the whole warp reaches the block barrier below together
  } else {
    // -------------------------------------------------------------- consumers
    const int ct = tid - 32;
    const int cw = warp - 1;
    int slot = 0;
    uint32_t phase = 0;
    while (true) {
      if (!mbar_wait_bounded(smem_u32(&full_bar[slot]), phase)) {
        atomicOr(&s_err, 1);
        break;
      }
      const StageDesc& ts = sdesc[slot];   // stays put until the slot is released
      if (ts.item < 0) break;
      const bool resid = ts.type == kDrawResid;
      int slot2 = slot + 1;
      uint32_t phase2 = phase;
      if (slot2 == kK3Stages) {
        slot2 = 0;
        phase2 ^= 1;
      }
      if (resid && !mbar_wait_bounded(smem_u32(&full_bar[slot2]), phase2)) {
        atomicOr(&s_err, 1);
        break;
      }
      const StageDesc& ds = resid ? sdesc[slot2] : ts;
      const int kc = ts.item % a.P;
      const int lo = kc * a.chunk_elems;
      const int hi = min(a.V, lo + a.chunk_elems);
      float sw, sp;
      if (resid)
        sum_stage<ES, true>(ts, ds, ring + slot * kK3SlotBytes, ring + slot2 * kK3SlotBytes, lo, hi, ct, a.c, sw, sp);
      else
        sum_stage<ES, false>(ts, ds, ring + slot * kK3SlotBytes, ring + slot * kK3SlotBytes, lo, hi, ct, a.c, sw, sp);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sw += __shfl_xor_sync(0xffffffffu, sw, o);
        sp += __shfl_xor_sync(0xffffffffu, sp, o);
      }
      int merger = 0;
      if (lane == 0) {
        red[slot][cw] = make_float2(sw, sp);
        __threadfence_block();
        merger = atomicAdd(&red_cnt[slot], 1) == kK3Consumers - 1;
      }
      if (__shfl_sync(0xffffffffu, merger, 0)) {
        __threadfence_block();
        float2 v = lane < kK3Consumers ? red[slot][lane] : make_float2(0.f, 0.f);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
          v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        }
        if (lane == 0) {
          atomicExch(&red_cnt[slot], 0);
          a.part[ts.item] = v;
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&empty_bar[slot]));
        if (resid) mbar_arrive(smem_u32(&empty_bar[slot2]));
      }
      slot = resid ? slot2 : slot;
      phase = resid ? phase2 : phase;
      if (++slot == kK3Stages) {
        slot = 0;
        phase ^= 1;
      }
    }
  }
  __syncthreads();
  if (s_err) {   // this CTA's sums are not to be trusted
    const float nan = __int_as_float(0x7fc00000);
    for (int64_t i = i0 + tid; i < i1; i += kK3Threads) a.part[i] = make_float2(nan, nan);
  }
}

// ------------------------------------------------------------------ K3b

__device__ __forceinline__ float2 chunk_sum(const float2* s_part, const float2* g_part, int k) {
  return k < kK3MaxChunks ? s_part[k] : __ldcg(&g_part[k]);
}

template <int ES>
__global__ void __launch_bounds__(kK3PickThreads) draw_pick_kernel(const DrawArgs a) {
  constexpr int E = kK3PickElems<ES>;
  constexpr int N = Elem<ES>::kVec;
  static_assert(E == N, "a pick thread owns one 16-byte vector of each row");
  constexpr int kWarps = kK3PickThreads / 32;
  __shared__ int s_stop_pre[kMaxStopIds];
  __shared__ float2 s_part[kK3MaxChunks];
  __shared__ int s_ex[kK3LocalExcl];
  __shared__ float scan_w[kWarps];
  __shared__ int s_chunk, s_usep, s_pick, s_lastpos;
  __shared__ float s_thr, s_S;
  __shared__ int s_fin[2];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  __shared__ FinishPre fpre;   // written by thread 0, read by thread 0 in finish_request
  if (a.fin_here) finish_prefetch(a.fin, b, s_stop_pre, fpre);
  grid_dep_wait();
  grid_dep_launch();

  // The descriptor, the chunk sums and the exclusion list, loaded together.
  const DrawDesc d = a.draws[b];
  const float2* pp_g = a.part + static_cast<int64_t>(b) * a.P;
  for (int k = tid; k < a.P && k < kK3MaxChunks; k += kK3PickThreads) s_part[k] = __ldcg(&pp_g[k]);
  const int32_t* gex = a.excl + static_cast<int64_t>(b) * a.excl_stride;
  if (tid < kK3LocalExcl && tid < a.excl_stride) s_ex[tid] = gex[tid];
  __syncthreads();
  if (d.type == kDrawNone) return;
  const bool resid = d.type == kDrawResid;
  const int nex = d.type == kDrawMaskedP ? d.n_excl : 0;
  const int* lst = nex <= kK3LocalExcl ? s_ex : gex;

  // Warp 0: the chunk holding u * S (fp32 warp scans, 32 chunks at a time;
  // the sums' rounding is far inside the 1e-5 * S band the comparison rules
  // allow at a boundary).
  if (warp == 0) {
    float sw = 0.f, sp = 0.f;
    for (int k = lane; k < a.P; k += 32) {
      const float2 v = chunk_sum(s_part, pp_g, k);
      sw += v.x;
      sp += v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sw += __shfl_xor_sync(0xffffffffu, sw, o);
      sp += __shfl_xor_sync(0xffffffffu, sp, o);
    }
    const int usep = !(sw > 0.f);
    const float S = usep ? sp : sw;
    const float thr = d.u * S;
    float run = 0.f, pre = 0.f, pre_last = 0.f;
    int cstar = -1, last_pos = -1;
    for (int base = 0; base < a.P; base += 32) {
      const int k = base + lane;
      float w = 0.f;
      if (k < a.P) {
        const float2 v = chunk_sum(s_part, pp_g, k);
        w = usep ? v.y : v.x;
      }
      float incl = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const float excl = run + (incl - w);
      const unsigned hit = __ballot_sync(0xffffffffu, k < a.P && excl + w > thr);
      if (cstar < 0 && hit) {
        const int l = __ffs(hit) - 1;
        cstar = base + l;
        pre = __shfl_sync(0xffffffffu, excl, l);
      }
      const unsigned pos = __ballot_sync(0xffffffffu, k < a.P && w > 0.f);
      if (pos) {   // last chunk with weight so far (the fallback when rounding leaves no crossing)
        const int l = 31 - __clz(pos);
        last_pos = base + l;
        pre_last = __shfl_sync(0xffffffffu, excl, l);
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (cstar < 0) {
      cstar = last_pos >= 0 ? last_pos : a.P - 1;
      pre = last_pos >= 0 ? pre_last : 0.f;
    }
    if (lane == 0) {
      s_chunk = cstar;
      s_usep = usep | (S == S ? 0 : 2);   // bit 1: a chunk sum was NaN (a wait gave up)
      s_thr = thr - pre;
      s_S = S;
      s_pick = INT_MAX;
      s_lastpos = -1;
    }
  }
  __syncthreads();

  // The chosen chunk: thread t owns elements [my0, my0 + E), one 16-byte
  // vector of each row where the row allows, and keeps them in registers.
  const int usep = s_usep & 1;
  const float thr = s_thr;
  const int lo2 = s_chunk * a.chunk_elems;
  const int hi2 = min(a.V, lo2 + a.chunk_elems);
  const int my0 = lo2 + tid * E;
  const uint8_t* trow = a.tgt + static_cast<int64_t>(d.t_row) * a.tgt_stride;
  const uint8_t* drow = resid ? a.dft + static_cast<int64_t>(d.d_row) * a.dft_stride : nullptr;
  float xs[E], ys[E];
  {
    const bool tvec = (reinterpret_cast<uintptr_t>(trow) & 15u) == 0 && my0 + E <= hi2;
    const bool dvec = !resid || ((reinterpret_cast<uintptr_t>(drow) & 15u) == 0 && my0 + E <= hi2);
    uint4 tq, dq;
    if (tvec) tq = __ldg(reinterpret_cast<const uint4*>(trow + static_cast<int64_t>(my0) * ES));
    if (resid && dvec) dq = __ldg(reinterpret_cast<const uint4*>(drow + static_cast<int64_t>(my0) * ES));
    if (tvec) {
      Elem<ES>::unpack(tq, xs);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) xs[e] = my0 + e < hi2 ? Elem<ES>::load(trow, my0 + e) : -INFINITY;
    }
    if (!resid) {
#pragma unroll
      for (int e = 0; e < E; ++e) ys[e] = 0.f;
    } else if (dvec) {
      Elem<ES>::unpack(dq, ys);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) ys[e] = my0 + e < hi2 ? Elem<ES>::load(drow, my0 + e) : -INFINITY;
    }
  }
  const uint32_t exm = (nex && !usep) ? excl_bits(my0, E, nex, lst) : 0u;
  float ws[E];
  float tsum = 0.f;
  int lastpos = -1;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float w = 0.f;
    if (my0 + e < hi2) {
      float p;
      weight_of(xs[e], ys[e], resid, a.c, d.lp2, d.lq2, w, p);
      if (usep) w = p;
      else if ((exm >> e) & 1u) w = 0.f;
      if (w > 0.f) lastpos = my0 + e;
    }
    ws[e] = w;
    tsum += w;
  }
  // Block exclusive scan of the per-thread sums (thread order = index order):
  // warp scans, then one warp scans the warp totals.
  float incl = tsum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) scan_w[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const float t = lane < kWarps ? scan_w[lane] : 0.f;
    float ti = t;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, ti, off);
      if (lane >= off) ti += v;
    }
    __syncwarp();
    if (lane < kWarps) scan_w[lane] = ti - t;
  }
  __syncthreads();
  const float excl_sum = scan_w[warp] + (incl - tsum);
  if (excl_sum + tsum > thr && tsum > 0.f) atomicMin(&s_pick, tid);
  if (lastpos >= 0) atomicMax(&s_lastpos, lastpos);
  __syncthreads();
  // The thread owning the drawn element: the crossing, else the last element
  // with weight, else the chunk's last element.
  int j_out = -1;
  if (s_pick != INT_MAX) {
    if (tid == s_pick) {
      float part = 0.f;
      bool found = false;
      j_out = lastpos;   // rounding left no crossing inside the thread
#pragma unroll
      for (int e = 0; e < E; ++e) {
        part += ws[e];
        if (!found && excl_sum + part > thr && ws[e] > 0.f) {
          j_out = my0 + e;
          found = true;
        }
      }
    }
  } else {
    const int jf = s_lastpos >= 0 ? s_lastpos : hi2 - 1;
    if (jf >= my0 && jf < my0 + E) j_out = jf;
  }
  if (j_out >= 0) {
    float x = 0.f, y = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (my0 + e == j_out) {
        x = xs[e];
        y = ys[e];
      }
    float w, p;
    weight_of(x, y, resid, a.c, d.lp2, d.lq2, w, p);
    const int64_t o = static_cast<int64_t>(b) * a.out_cols + d.pos;
    a.out_tokens[o] = j_out;
    if (a.out_logprob) a.out_logprob[o] = (x * a.c - d.lp2) * kLn2;
    if (a.out_mu) a.out_mu[o] = d.type == kDrawMaskedP ? d.scale * p / s_S : p;
    if ((s_usep & 2) && a.out_status) atomicOr(&a.out_status[b], kStatusWaitErr);
  }
  if (a.fin_here) {   // no mu pass follows: this kernel ends the call
    __syncthreads();
    finish_request(a.fin, fpre, s_stop_pre, b, d.pos, a.out_cols, a.out_tokens, a.out_logprob, a.out_mu, a.out_nodes,
                   a.out_status, s_fin);
  }
}

}  // namespace sv
