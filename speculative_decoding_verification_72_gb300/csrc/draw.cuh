// K3: the one draw per request that ends a stochastic round (spec-decode
// README, "How it works": on the first rejection a sample from
// normalize(relu(p - q)); after K acceptances a bonus sample from p; the
// nanospec README's tree and deterministic-draft rules draw from p with the
// rejected tokens removed).
//
// Grid = B x P CTAs; CTA (b, c) sums the weights w_j of vocabulary chunk c
// (kK3ChunkElems elements) of request b's row (and, for the zero-mass
// fallback, sum p_j) with coalesced element-strided loads, and takes a
// ticket. The last CTA of request b forms the ordered prefix over the P chunk
// sums in double, finds the chunk where u * S falls, recomputes that chunk's
// weights (just read, so L2-resident) into shared memory, and resolves the
// smallest j whose inclusive prefix sum exceeds u * S with a block scan over
// contiguous shared-memory segments. Per-element weights are recomputed by the
// same code in both passes.
#pragma once

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

__device__ __forceinline__ float2 chunk_sum(const float2* s_part, const float2* g_part, int k) {
  return k < kK3MaxChunks ? s_part[k] : __ldcg(&g_part[k]);
}

struct DrawArgs {
  const uint8_t* tgt;
  int64_t tgt_stride;   // bytes
  const uint8_t* dft;
  int64_t dft_stride;   // bytes
  int32_t V, P, chunk_elems;
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

template <int ES>
__global__ void __launch_bounds__(kK3Threads) draw_kernel(const DrawArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float red[kK3Threads / 32];
  __shared__ float scan_w[kK3Threads / 32];
  __shared__ float seg[kK3Threads * kK3SegStride];
  __shared__ int s_ex[kK3LocalExcl];
  __shared__ int s_nex;
  __shared__ int s_last, s_chunk, s_usep, s_pick, s_lastpos;
  __shared__ float s_thr;
  __shared__ double s_S;
  __shared__ float2 s_part[kK3MaxChunks];

  const int tid = threadIdx.x;
  const int b = blockIdx.x / a.P;
  const int ch = blockIdx.x - b * a.P;
  const DrawDesc d = a.draws[b];
  if (d.type == kDrawNone) return;
  const int32_t* ex = a.excl + static_cast<int64_t>(b) * a.excl_stride;
  DrawRow<ES> row;
  row.t = a.tgt + static_cast<int64_t>(d.t_row) * a.tgt_stride;
  row.d = d.type == kDrawResid ? a.dft + static_cast<int64_t>(d.d_row) * a.dft_stride : nullptr;
  row.c = a.c;
  row.lp2 = d.lp2;
  row.lq2 = d.lq2;

  // Pass 1: this chunk's weight sums (element j = lo + tid + k * kK3Threads).
  const int lo = ch * a.chunk_elems;
  const int hi = min(a.V, lo + a.chunk_elems);
  int nex = gather_excl(d, ex, lo, hi, s_ex, &s_nex);
  float sw = 0.f, sp = 0.f;
#pragma unroll
  for (int k = 0; k < kK3PerThread; ++k) {
    const int j = lo + tid + k * kK3Threads;
    if (j < hi) {
      float w, p;
      row.weight(j, w, p);
      if (nex && is_excluded(j, nex, s_ex, ex, d.n_excl)) w = 0.f;
      sw += w;
      sp += p;
    }
  }
  const float tw = block_sum_fixed(sw, red);
  const float tp = block_sum_fixed(sp, red);
  if (tid == 0) {
    a.part[static_cast<int64_t>(b) * a.P + ch] = make_float2(tw, tp);
    __threadfence();
    const uint32_t ticket = atomicAdd(&a.counters[b], 1u);
    s_last = (ticket == static_cast<uint32_t>(a.P - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last CTA of request b: the chunk sums are loaded together into shared
  // memory (a loop of dependent loads would pay one L2 round trip per
  // chunk), then thread 0 forms their ordered prefix in double.
  const float2* pp_g = a.part + static_cast<int64_t>(b) * a.P;
  for (int k = tid; k < a.P && k < kK3MaxChunks; k += kK3Threads) s_part[k] = __ldcg(&pp_g[k]);
  __syncthreads();
  if (tid == 0) {
    double S = 0.0;
    for (int k = 0; k < a.P; ++k) S += static_cast<double>(chunk_sum(s_part, pp_g, k).x);
    int usep = !(S > 0.0);
    if (usep) {
      S = 0.0;
      for (int k = 0; k < a.P; ++k) S += static_cast<double>(chunk_sum(s_part, pp_g, k).y);
    }
    const double thr = static_cast<double>(d.u) * S;
    double pre = 0.0;
    int cstar = -1;
    for (int k = 0; k < a.P; ++k) {
      const float2 v = chunk_sum(s_part, pp_g, k);
      const double w = usep ? v.y : v.x;
      if (pre + w > thr) {
        cstar = k;
        break;
      }
      pre += w;
    }
    if (cstar < 0) {   // rounding left no crossing: last chunk with weight
      double run = 0.0, pre_last = 0.0;
      for (int k = 0; k < a.P; ++k) {
        const float2 v = chunk_sum(s_part, pp_g, k);
        const double w = usep ? v.y : v.x;
        if (w > 0.0) {
          cstar = k;
          pre_last = run;
        }
        run += w;
      }
      pre = pre_last;
      if (cstar < 0) cstar = a.P - 1;
    }
    s_chunk = cstar;
    s_usep = usep;
    s_thr = static_cast<float>(thr - pre);
    s_S = S;
    s_pick = INT_MAX;
    s_lastpos = -1;
    a.counters[b] = 0u;
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
#pragma unroll
  for (int k = 0; k < kK3PerThread; ++k) {
    const int i = tid + k * kK3Threads;   // chunk offset
    const int j = lo2 + i;
    float w = 0.f;
    if (j < hi2) {
      float p;
      row.weight(j, w, p);
      if (usep) w = p;
      else if (nex && is_excluded(j, nex, s_ex, ex, d.n_excl)) w = 0.f;
    }
    seg[(i / kK3PerThread) * kK3SegStride + (i % kK3PerThread)] = w;
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
      if (d.type == kDrawMaskedP) mu = static_cast<float>(static_cast<double>(d.scale) * p / s_S);
      a.out_mu[o] = mu;
    }
  }
}

}  // namespace sv
