// K3: the one draw per request that ends a stochastic round (spec-decode
// README, "How it works": on the first rejection a sample from
// normalize(relu(p - q)); after K acceptances a bonus sample from p; the
// nanospec README's tree and deterministic-draft rules draw from p with the
// rejected tokens removed).
//
// Grid = B x Q CTAs; CTA (b, q) sums the weights w_j of vocabulary chunks
// q*cpc .. q*cpc + cpc - 1 (kK3ChunkElems elements each) of request b's row
// (and, for the zero-mass fallback, sum p_j), one sum pair per chunk, and
// takes a ticket. Chunks are read two at a time with every load of the pair
// issued before any arithmetic: 16-byte vectors when both rows are 16-byte
// aligned and the CTA's range holds no removed token, else element-strided
// scalars. The last CTA of request b forms the ordered prefix over the P chunk
// sums (one warp, fp32 scans), finds the chunk where u * S falls, recomputes that chunk's
// weights (just read, so L2-resident) into shared memory, and resolves the
// smallest j whose inclusive prefix sum exceeds u * S with a block scan over
// contiguous shared-memory segments. Per-element weights are recomputed by the
// same code in both passes.
#pragma once

#include "finish.cuh"
#include "sv_common.cuh"

namespace sv {

constexpr int kK3Threads = 256;
constexpr int kK3PerThread = 16;                          // elements per thread per chunk
constexpr int kK3ChunkElems = kK3Threads * kK3PerThread;  // 4096
constexpr int kK3SegStride = kK3PerThread + 1;           // padded shared-memory segment
constexpr int kK3LocalExcl = 64;
// Chunk sums staged in shared memory by the last CTA (V up to 1M elements;
// beyond that the rest are read from global memory).
constexpr int kK3MaxChunks = 256;
// Chunks one CTA sums in pass 1: its loads for all of them are in flight at
// once (64 data registers per thread for fp32 with draft rows).
template <int ES>
constexpr int kK3Cpc = ES == 2 ? 4 : 2;
constexpr int kK3MaxCpc = 4;

__device__ __forceinline__ float2 chunk_sum(const float2* s_part, const float2* g_part, int k) {
  return k < kK3MaxChunks ? s_part[k] : __ldcg(&g_part[k]);
}

struct DrawArgs {
  const uint8_t* tgt;
  int64_t tgt_stride;   // bytes
  const uint8_t* dft;
  int64_t dft_stride;   // bytes
  int32_t V, P, chunk_elems;
  int32_t Q;            // CTAs per request: ceil(P / kK3Cpc<ES>)
  float c;              // log2(e) / T
  const DrawDesc* draws;
  const int32_t* excl;
  int32_t excl_stride;
  float2* part;         // [B * P]: (sum w, sum p)
  uint32_t* counters;   // [B], zeroed by K2 of the same call
  int32_t out_cols;
  int32_t* out_tokens;
  float* out_logprob;
  float* out_mu;
  int32_t* out_nodes;    // tree calls, else nullptr
  int32_t* out_status;
  FinishArgs fin;        // applied by the last CTA of a request when fin_here
  int32_t fin_here;
};

template <int ES>
struct DrawRow {
  const uint8_t* t;
  const uint8_t* d;   // nullptr unless kDrawResid
  float c, lp2, lq2;
  __device__ __forceinline__ void weight(int j, float& w, float& p) const {
    const float x = Elem<ES>::load(t, j);
    p = ex2(fmaf(x, c, -lp2));
    if (d) {
      const float q = ex2(fmaf(Elem<ES>::load(d, j), c, -lq2));
      w = fmaxf(p - q, 0.f);
    } else {
      w = p;
    }
  }
};

__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kK3Threads / 32; ++w) t += red[w];
  return t;   // valid in thread 0
}

// Load the exclusions that fall in [lo, hi) into shared memory; returns the
// count (a value above kK3LocalExcl means "use the global list").
__device__ __forceinline__ int gather_excl(const DrawDesc& d, const int32_t* ex, int lo, int hi,
                                           int* s_ex, int* s_nex) {
  __syncthreads();
  if (threadIdx.x == 0) *s_nex = 0;
  __syncthreads();
  if (d.type == kDrawMaskedP) {
    for (int k = threadIdx.x; k < d.n_excl; k += kK3Threads) {
      const int t = ex[k];
      if (t >= lo && t < hi) {
        const int slot = atomicAdd(s_nex, 1);
        if (slot < kK3LocalExcl) s_ex[slot] = t;
      }
    }
  }
  __syncthreads();
  return *s_nex;
}

__device__ __forceinline__ bool is_excluded(int j, int nex, const int* s_ex, const int32_t* ex,
                                            int n_all) {
  if (nex == 0) return false;
  if (nex <= kK3LocalExcl) {
    for (int k = 0; k < nex; ++k)
      if (s_ex[k] == j) return true;
    return false;
  }
  for (int k = 0; k < n_all; ++k)
    if (ex[k] == j) return true;
  return false;
}

// Weights of one element from its logits (same arithmetic as DrawRow::weight).
__device__ __forceinline__ void weight_of(float x, float y, bool resid, float c, float lp2, float lq2,
                                          float& w, float& p) {
  p = ex2(fmaf(x, c, -lp2));
  w = resid ? fmaxf(p - ex2(fmaf(y, c, -lq2)), 0.f) : p;
}

// Pass 1 of one CTA: the (w, p) sums of its kK3Cpc<ES> chunks c0, c0 + 1, ...
// (those below c_end), in acc[2 * i], acc[2 * i + 1]. When both rows are
// 16-byte aligned every load is issued before any arithmetic, so a CTA pays
// one memory round trip (16-byte vectors, chunk-relative vector
// t + k * kK3Threads of thread t; the row's last partial vector element by
// element). A vector holding a removed token is left out of that loop and
// summed afterwards element by element. Unaligned rows take element-strided
// scalar loads, one chunk at a time.
template <int ES>
struct Pass1 {
  static constexpr int N = Elem<ES>::kVec;
  static constexpr int VPT = kK3ChunkElems / N / kK3Threads;   // vectors per thread per chunk
  static constexpr int C = kK3Cpc<ES>;

  __device__ __forceinline__ static void vec(const DrawRow<ES>& row, int c0, int c_end, int V, int chunk,
                                             int nex, const int* s_ex, const int32_t* ex, int n_all,
                                             float (&acc)[2 * C]) {
    const bool resid = row.d != nullptr;
    uint4 xv[C][VPT], yv[C][VPT];
    const uint4* tv = reinterpret_cast<const uint4*>(row.t + static_cast<int64_t>(c0) * chunk * ES);
    const uint4* dv = resid ? reinterpret_cast<const uint4*>(row.d + static_cast<int64_t>(c0) * chunk * ES) : nullptr;
    const int nfull = (min(V, c_end * chunk) - c0 * chunk) / N;   // whole vectors in the range
    constexpr int kChunkVecs = kK3ChunkElems / N;
    // Bit i * VPT + k: this thread's vector k of chunk c0 + i holds a removed token.
    uint32_t exmask = 0u;
    if (nex) {
      const int n_list = nex <= kK3LocalExcl ? nex : n_all;
      for (int r = 0; r < n_list; ++r) {
        const int v = ((nex <= kK3LocalExcl ? s_ex[r] : ex[r]) - c0 * chunk);
        if (v < 0 || v >= nfull * N) continue;
        const int vv = v / N, i = vv / kChunkVecs, vc = vv - i * kChunkVecs;
        if (vc % kK3Threads == static_cast<int>(threadIdx.x)) exmask |= 1u << (i * VPT + vc / kK3Threads);
      }
    }
#pragma unroll
    for (int i = 0; i < C; ++i) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = i * kChunkVecs + static_cast<int>(threadIdx.x) + k * kK3Threads;
        xv[i][k] = make_uint4(0u, 0u, 0u, 0u);
        yv[i][k] = make_uint4(0u, 0u, 0u, 0u);
        if (v < nfull) {
          xv[i][k] = __ldg(tv + v);
          if (resid) yv[i][k] = __ldg(dv + v);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < C; ++i) {
      float sw = 0.f, sp = 0.f;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (i * kChunkVecs + static_cast<int>(threadIdx.x) + k * kK3Threads < nfull &&
            !((exmask >> (i * VPT + k)) & 1u)) {
          float xf[N], yf[N];
          Elem<ES>::unpack(xv[i][k], xf);
          Elem<ES>::unpack(yv[i][k], yf);
#pragma unroll
          for (int e = 0; e < N; ++e) {
            float w, p;
            weight_of(xf[e], yf[e], resid, row.c, row.lp2, row.lq2, w, p);
            sw += w;
            sp += p;
          }
        }
      }
      acc[2 * i] = sw;
      acc[2 * i + 1] = sp;
    }
    // vectors holding a removed token, element by element
#pragma unroll 1
    while (exmask) {
      const int bit = __ffs(exmask) - 1;
      exmask &= exmask - 1u;
      const int i = bit / VPT, k = bit - i * VPT;
      const int j0 = (c0 + i) * chunk + (static_cast<int>(threadIdx.x) + k * kK3Threads) * N;
      float sw = 0.f, sp = 0.f;
#pragma unroll 1
      for (int e = 0; e < N; ++e) {
        float w, p;
        row.weight(j0 + e, w, p);
        if (is_excluded(j0 + e, nex, s_ex, ex, n_all)) w = 0.f;
        sw += w;
        sp += p;
      }
#pragma unroll
      for (int q = 0; q < C; ++q)
        if (q == i) {
          acc[2 * q] += sw;
          acc[2 * q + 1] += sp;
        }
    }
    // elements after the last whole vector (fewer than N), in the last chunk
    const int jt = c0 * chunk + nfull * N + static_cast<int>(threadIdx.x);
    if (static_cast<int>(threadIdx.x) < N && jt < min(V, c_end * chunk)) {
      float w, p;
      row.weight(jt, w, p);
      if (nex && is_excluded(jt, nex, s_ex, ex, n_all)) w = 0.f;
      const int i = (jt - c0 * chunk) / chunk;
#pragma unroll
      for (int q = 0; q < C; ++q)
        if (q == i) {
          acc[2 * q] += w;
          acc[2 * q + 1] += p;
        }
    }
  }

  // Scalar variant, one chunk at a time: element j = chunk start + t + k * kK3Threads.
  __device__ __forceinline__ static void scalar(const DrawRow<ES>& row, int c0, int c_end, int V, int chunk,
                                                int nex, const int* s_ex, const int32_t* ex, int n_all,
                                                float (&acc)[2 * C]) {
    const bool resid = row.d != nullptr;
#pragma unroll
    for (int q = 0; q < 2 * C; ++q) acc[q] = 0.f;
#pragma unroll 1
    for (int i = 0; i < C && c0 + i < c_end; ++i) {
      const int lo = (c0 + i) * chunk, hi = min(V, lo + chunk);
      float xs[kK3PerThread], ys[kK3PerThread];
#pragma unroll
      for (int k = 0; k < kK3PerThread; ++k) {
        const int j = lo + static_cast<int>(threadIdx.x) + k * kK3Threads;
        xs[k] = -INFINITY;
        ys[k] = -INFINITY;
        if (j < hi) {
          xs[k] = Elem<ES>::load(row.t, j);
          if (resid) ys[k] = Elem<ES>::load(row.d, j);
        }
      }
      float sw = 0.f, sp = 0.f;
#pragma unroll
      for (int k = 0; k < kK3PerThread; ++k) {
        const int j = lo + static_cast<int>(threadIdx.x) + k * kK3Threads;
        if (j < hi) {
          float w, p;
          weight_of(xs[k], ys[k], resid, row.c, row.lp2, row.lq2, w, p);
          if (nex && is_excluded(j, nex, s_ex, ex, n_all)) w = 0.f;
          sw += w;
          sp += p;
        }
      }
#pragma unroll
      for (int q = 0; q < C; ++q)
        if (q == i) {
          acc[2 * q] = sw;
          acc[2 * q + 1] = sp;
        }
    }
  }
};

// Reduce 2 * C per-thread values over the CTA (fixed order); valid in thread 0.
template <int C>
__device__ __forceinline__ void block_sum_n(float (&v)[2 * C], float* red_n) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int q = 0; q < 2 * C; ++q) v[q] += __shfl_down_sync(0xffffffffu, v[q], off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int q = 0; q < 2 * C; ++q) red_n[warp * 2 * C + q] = v[q];
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int q = 0; q < 2 * C; ++q) {
      float t = 0.f;
      for (int w = 0; w < kK3Threads / 32; ++w) t += red_n[w * 2 * C + q];
      v[q] = t;
    }
  }
}

template <int ES>
__global__ void __launch_bounds__(kK3Threads) draw_kernel(const DrawArgs a) {
  __shared__ int s_stop_pre[kMaxStopIds];
  FinishPre fpre;
  if (a.fin_here) finish_prefetch(a.fin, blockIdx.x / a.Q, s_stop_pre, fpre);
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float red_n[kK3Threads / 32 * 2 * kK3MaxCpc];
  __shared__ float scan_w[kK3Threads / 32];
  __shared__ float seg[kK3Threads * kK3SegStride];
  __shared__ int s_ex[kK3LocalExcl];
  __shared__ int s_nex;
  __shared__ int s_last, s_chunk, s_usep, s_pick, s_lastpos;
  __shared__ float s_thr;
  __shared__ float s_S;
  __shared__ float2 s_part[kK3MaxChunks];
  __shared__ int s_fin[2];

  const int tid = threadIdx.x;
  const int b = blockIdx.x / a.Q;
  const int q = blockIdx.x - b * a.Q;
  const DrawDesc d = a.draws[b];
  if (d.type == kDrawNone) return;
  const int32_t* ex = a.excl + static_cast<int64_t>(b) * a.excl_stride;
  DrawRow<ES> row;
  row.t = a.tgt + static_cast<int64_t>(d.t_row) * a.tgt_stride;
  row.d = d.type == kDrawResid ? a.dft + static_cast<int64_t>(d.d_row) * a.dft_stride : nullptr;
  row.c = a.c;
  row.lp2 = d.lp2;
  row.lq2 = d.lq2;

  // Pass 1: the weight sums of this CTA's chunks.
  constexpr int C = kK3Cpc<ES>;
  const int c0 = q * C;
  const int c1 = min(a.P, c0 + C);
  const int lo = c0 * a.chunk_elems;
  const int hi = min(a.V, c1 * a.chunk_elems);
  int nex = gather_excl(d, ex, lo, hi, s_ex, &s_nex);
  const bool vec = (reinterpret_cast<uintptr_t>(row.t) & 15u) == 0 &&
                   (row.d == nullptr || (reinterpret_cast<uintptr_t>(row.d) & 15u) == 0);
  float acc[2 * C];
  if (vec) Pass1<ES>::vec(row, c0, c1, a.V, a.chunk_elems, nex, s_ex, ex, d.n_excl, acc);
  else Pass1<ES>::scalar(row, c0, c1, a.V, a.chunk_elems, nex, s_ex, ex, d.n_excl, acc);
  block_sum_n<C>(acc, red_n);
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < C; ++i)
      if (c0 + i < c1) a.part[static_cast<int64_t>(b) * a.P + c0 + i] = make_float2(acc[2 * i], acc[2 * i + 1]);
  }
  if (tid == 0) {
    __threadfence();
    const uint32_t ticket = atomicAdd(&a.counters[b], 1u);
    s_last = (ticket == static_cast<uint32_t>(a.Q - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last CTA of request b: the chunk sums are loaded together into shared
  // memory (a loop of dependent loads would pay one L2 round trip per
  // chunk), then warp 0 finds the chunk holding u * S with fp32 warp scans,
  // 32 chunks at a time (a serial fp64 prefix here cost ~9 us: FP64 latency
  // is long on this GPU). fp32 adds at most a few ulps of S, far inside the
  // 1e-5 * S band the comparison rules allow at a boundary.
  const float2* pp_g = a.part + static_cast<int64_t>(b) * a.P;
  for (int k = tid; k < a.P && k < kK3MaxChunks; k += kK3Threads) s_part[k] = __ldcg(&pp_g[k]);
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
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
      s_usep = usep;
      s_thr = thr - pre;
      s_S = S;
      s_pick = INT_MAX;
      s_lastpos = -1;
      a.counters[b] = 0u;
    }
  }
  __syncthreads();

  // Pass 2: the chosen chunk's weights into shared memory (coalesced), then a
  // scan over contiguous segments: thread t owns elements [t*16, t*16 + 16).
  const int c2 = s_chunk;
  const int usep = s_usep;
  const float thr = s_thr;
  const int lo2 = c2 * a.chunk_elems;
  const int hi2 = min(a.V, lo2 + a.chunk_elems);
  nex = usep ? 0 : gather_excl(d, ex, lo2, hi2, s_ex, &s_nex);
  {
    float xs[kK3PerThread], ys[kK3PerThread];   // loads first, all in flight together
#pragma unroll
    for (int k = 0; k < kK3PerThread; ++k) {
      const int j = lo2 + tid + k * kK3Threads;
      xs[k] = -INFINITY;
      ys[k] = -INFINITY;
      if (j < hi2) {
        xs[k] = Elem<ES>::load(row.t, j);
        if (row.d) ys[k] = Elem<ES>::load(row.d, j);
      }
    }
#pragma unroll
    for (int k = 0; k < kK3PerThread; ++k) {
      const int i = tid + k * kK3Threads;   // chunk offset
      const int j = lo2 + i;
      float w = 0.f;
      if (j < hi2) {
        float p;
        weight_of(xs[k], ys[k], row.d != nullptr, row.c, row.lp2, row.lq2, w, p);
        if (usep) w = p;
        else if (nex && is_excluded(j, nex, s_ex, ex, d.n_excl)) w = 0.f;
      }
      seg[(i / kK3PerThread) * kK3SegStride + (i % kK3PerThread)] = w;
    }
  }
  __syncthreads();
  const float* mine = seg + tid * kK3SegStride;
  float tsum = 0.f;
  int lastpos = -1;
#pragma unroll
  for (int k = 0; k < kK3PerThread; ++k) {
    tsum += mine[k];
    if (mine[k] > 0.f) lastpos = lo2 + tid * kK3PerThread + k;
  }
  // Block exclusive scan of the per-thread sums (thread order = index order).
  const int warp = tid >> 5, lane = tid & 31;
  float incl = tsum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) scan_w[warp] = incl;
  __syncthreads();
  float wbase = 0.f;
  for (int w = 0; w < warp; ++w) wbase += scan_w[w];
  const float excl_sum = wbase + incl - tsum;
  if (excl_sum + tsum > thr && tsum > 0.f) atomicMin(&s_pick, tid);
  if (lastpos >= 0) atomicMax(&s_lastpos, lastpos);
  __syncthreads();
  int j_out = -1;
  if (s_pick == INT_MAX) {
    if (tid == 0) j_out = s_lastpos >= 0 ? s_lastpos : hi2 - 1;
  } else if (tid == s_pick) {
    float part = 0.f;
    j_out = lastpos;
#pragma unroll
    for (int k = 0; k < kK3PerThread; ++k) {
      part += mine[k];
      if (excl_sum + part > thr && mine[k] > 0.f) {
        j_out = lo2 + tid * kK3PerThread + k;
        break;
      }
    }
  }
  if (j_out >= 0) {
    float w, p;
    row.weight(j_out, w, p);
    const float x = Elem<ES>::load(row.t, j_out);
    const int64_t o = static_cast<int64_t>(b) * a.out_cols + d.pos;
    a.out_tokens[o] = j_out;
    if (a.out_logprob) a.out_logprob[o] = (x * a.c - d.lp2) * kLn2;
    if (a.out_mu) {
      float mu = p;
      if (d.type == kDrawMaskedP) mu = d.scale * p / s_S;
      a.out_mu[o] = mu;
    }
  }
  if (a.fin_here) {   // no mu pass follows: this kernel ends the call
    __syncthreads();
    finish_request(a.fin, fpre, s_stop_pre, b, d.pos, a.out_cols, a.out_tokens, a.out_logprob, a.out_mu, a.out_nodes,
                   a.out_status, s_fin);
  }
}

}  // namespace sv
