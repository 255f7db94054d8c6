// Kernels that only the relaxed and power acceptance rules need (nanospec
// README, acceptance rules):
//
// topk_threshold_kernel
//   The relaxed rule accepts t when p(t) >= tau or rank(t) < k, with rank(t)
//   the number of logits strictly greater than x_t. rank(t) < k holds exactly
//   when x_t >= v_k, the k-th largest logit of the row counted with
//   multiplicity (if x_t >= v_k, only elements above v_k can exceed x_t, and
//   there are fewer than k of them; if x_t < v_k, the k largest all exceed
//   it). So the rank test needs one number per row, whatever tokens the row
//   scores. v_k is found by a most-significant-digit radix select over
//   order-preserving integer keys of the raw logits, 8 bits per pass (2
//   passes for bf16, 4 for fp32), one CTA per row. Tree rows without a child
//   are skipped.
//
// mu_pass_kernel
//   With draft logits, the power and relaxed rules accept draft t with
//   acc(t) = min(1, p/q)^alpha or [p >= tau or rank < k], and a rejection at
//   row n draws from normalize(relu(p_n - q_n)). The sampler's probability of
//   emitting a at row j is then
//       mu_j(a) = q_j(a) acc_j(a) + (1 - keep_j) res_j(a),
//       keep_j = sum_s q_j(s) acc_j(s),  res_j = relu(p_j - q_j) / sum relu(p_j - q_j)
//   (res_j = p_j when that mass is zero), which needs two full-row sums per
//   emitted draft row. Grid = B x K x P CTAs; CTA (b, j, c) sums vocabulary
//   chunk c of row j when j <= n_b, then takes a ticket; the last CTA of
//   request b adds the chunk sums in order and writes mu for
//   positions 0..min(n_b, K-1), reading the draw at position n_b from K3's
//   output.
#pragma once

#include "decide.cuh"
#include "draw.cuh"

namespace sv {

// ------------------------------------------------------------ top-k bound

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;

// Order-preserving keys: key(a) < key(b) iff a < b for non-NaN a, b (with
// -0 below +0, which leaves every threshold compare unchanged).
template <int ES>
struct KeyOf;

template <>
struct KeyOf<4> {
  static constexpr int kBits = 32;
  __device__ __forceinline__ static uint32_t key(const uint8_t* row, int j) {
    const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(row) + j);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }
  __device__ __forceinline__ static float value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
  }
};

template <>
struct KeyOf<2> {
  static constexpr int kBits = 16;
  __device__ __forceinline__ static uint32_t key(const uint8_t* row, int j) {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned short*>(row) + j);
    return (u & 0x8000u) ? (~u & 0xffffu) : (u | 0x8000u);
  }
  __device__ __forceinline__ static float value(uint32_t k) {
    const uint32_t u = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
    return __uint_as_float(u << 16);
  }
};

struct TopkArgs {
  const uint8_t* tgt;
  int64_t tgt_stride;      // bytes
  int32_t rows_per_req;    // rows that may be tested per request (chain K, tree N)
  int32_t row_pitch;       // target rows per request (chain K+1, tree N)
  int32_t V, k;
  const int32_t* parents;  // tree: [B, N]; chain: nullptr
  float* thr;              // [B * rows_per_req]: v_k, +inf for skipped rows
};

template <int ES>
__global__ void __launch_bounds__(kTkThreads) topk_threshold_kernel(const TopkArgs a) {
  __shared__ uint32_t hist[kTkWarps][256];
  __shared__ uint32_t tot[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_k;
  // Wait for the kernel before (K1) to complete: the decide kernel after this
  // one waits only for this grid, and reads K1's results.
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x / a.rows_per_req;
  const int j = blockIdx.x - b * a.rows_per_req;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (a.parents) {   // a tree row is tested only if some node links to it
    const int32_t* par = a.parents + static_cast<int64_t>(b) * a.rows_per_req;
    bool has = false;
    for (int c = j + 1 + tid; c < a.rows_per_req; c += kTkThreads) has |= (par[c] == j);
    if (!__syncthreads_or(has)) {
      if (tid == 0) a.thr[blockIdx.x] = INFINITY;
      return;
    }
  }
  const uint8_t* row = a.tgt + (static_cast<int64_t>(b) * a.row_pitch + j) * a.tgt_stride;
  uint32_t prefix = 0;   // key digits fixed so far
  int kr = min(a.k, a.V);   // rank still to find among the keys matching prefix
#pragma unroll 1
  for (int pass = 0; pass < KeyOf<ES>::kBits / 8; ++pass) {
    const int shift = KeyOf<ES>::kBits - 8 * (pass + 1);
    for (int i = tid; i < kTkWarps * 256; i += kTkThreads) (&hist[0][0])[i] = 0u;
    __syncthreads();
    // Uniform trip count per warp, so the match below sees all 32 lanes.
    for (int base = 0; base < a.V; base += kTkThreads) {
      const int e = base + tid;
      uint32_t bin = 256u;
      if (e < a.V) {
        const uint32_t key = KeyOf<ES>::key(row, e);
        if (pass == 0 || (key >> (shift + 8)) == prefix) bin = (key >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin < 256u && lane == __ffs(peers) - 1) atomicAdd(&hist[warp][bin], __popc(peers));
    }
    __syncthreads();
    for (int i = tid; i < 256; i += kTkThreads) {
      uint32_t s = 0;
#pragma unroll
      for (int w = 0; w < kTkWarps; ++w) s += hist[w][i];
      tot[i] = s;
    }
    __syncthreads();
    if (warp == 0) {
      // Lane l holds digits 255-8l down to 248-8l; an inclusive scan over
      // lanes counts the keys at or above each lane's lowest digit.
      uint32_t cnt[8];
      uint32_t ls = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        cnt[q] = tot[255 - 8 * lane - q];
        ls += cnt[q];
      }
      uint32_t incl = ls;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      uint32_t run = incl - ls;
      const uint32_t want = static_cast<uint32_t>(kr);
      if (run < want && want <= incl) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (run + cnt[q] >= want) {
            s_prefix = (prefix << 8) | static_cast<uint32_t>(255 - 8 * lane - q);
            s_k = static_cast<int>(want - run);
            break;
          }
          run += cnt[q];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    kr = s_k;
  }
  if (tid == 0) a.thr[blockIdx.x] = KeyOf<ES>::value(prefix);
}

// ----------------------------------------------------------- mu pass

constexpr int kMuThreads = 256;

// Sum over the CTA in a fixed order; the result is valid in thread 0.
__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_down_sync(0xffffffffu, v, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kMuThreads / 32; ++w) t += red[w];
  return t;
}

struct MuArgs {
  const uint8_t* tgt;
  int64_t tgt_stride;      // bytes
  const uint8_t* dft;
  int64_t dft_stride;      // bytes
  const int32_t* drafts;   // [B, K]
  int32_t B, K, V, P, chunk_elems;
  const Partial* part;     // K1 partials: target rows, then draft rows
  int64_t T;
  int32_t G;
  float c;
  RuleArgs rule;           // rule.thr: [B * K] relaxed rank bound, or nullptr
  const int32_t* num;      // n per request (decide kernel)
  const int32_t* tokens;   // [B, K+1]: the draw at position n (draw kernel)
  float* out_mu;           // [B, K+1]
  int32_t* out_tokens;     // [B, K+1] (the same array as tokens; cleared by the finish step)
  float* out_logprob;
  int32_t* out_status;
  FinishArgs fin;          // stop / cap / counters, applied by the last CTA of a request
  float2* mpart;           // [B * K * P]: (sum q acc, sum relu(p - q))
  uint32_t* counters;      // [B], zeroed by the decide kernel of the same call
};

// q(s) acc(s) for one vocabulary entry, in the log2 domain:
// lp = log2 p(s), lq = log2 q(s), x = the raw target logit.
__device__ __forceinline__ float kept_mass(const RuleArgs& r, float lp, float lq, float x, float thr) {
  if (lq == -INFINITY) return 0.f;
  if (r.rule == 1) return relaxed_accepts(r, lp, x, thr) ? ex2(lq) : 0.f;
  // power: q min(1, p/q)^alpha = q when p >= q, else 2^(lq + alpha (lp - lq))
  return ex2(lp >= lq ? lq : fmaf(r.alpha, lp - lq, lq));
}

template <int ES>
__device__ __forceinline__ void row_lse2(const MuArgs& a, int b, int j, float& lp2, float& lq2) {
  float m, s;
  int idx, err;
  merge_row_serial(a.part, static_cast<int64_t>(b) * (a.K + 1) + j, a.V, a.T, a.G, a.c, m, s, idx, err);
  lp2 = m * a.c + log2f(s);
  merge_row_serial(a.part, static_cast<int64_t>(a.B) * (a.K + 1) + static_cast<int64_t>(b) * a.K + j, a.V, a.T,
            a.G, a.c, m, s, idx, err);
  lq2 = m * a.c + log2f(s);
}

template <int ES>
__global__ void __launch_bounds__(kMuThreads) mu_pass_kernel(const MuArgs a) {
  __shared__ float red[kMuThreads / 32];
  __shared__ float s_lp2, s_lq2;
  __shared__ int s_last, s_fin[2];
  __shared__ int s_stop[kMaxStopIds];
  const int per_req = a.K * a.P;
  __shared__ FinishPre fpre;   // written by thread 0, read by thread 0 in finish_request
  finish_prefetch(a.fin, blockIdx.x / per_req, s_stop, fpre);
  grid_dep_wait();
  grid_dep_launch();
  const int tid = threadIdx.x;
  const int b = blockIdx.x / per_req;
  const int r = blockIdx.x - b * per_req;
  const int j = r / a.P;
  const int ch = r - j * a.P;
  const int n = a.num[b];
  const float thr_row = a.rule.thr ? a.rule.thr[static_cast<int64_t>(b) * a.K + j] : INFINITY;

  if (j <= n) {   // rows after the decision are not emitted
    if (tid == 0) row_lse2<ES>(a, b, j, s_lp2, s_lq2);
    __syncthreads();
    const float lp2 = s_lp2, lq2 = s_lq2;
    const uint8_t* trow = a.tgt + (static_cast<int64_t>(b) * (a.K + 1) + j) * a.tgt_stride;
    const uint8_t* drow = a.dft + (static_cast<int64_t>(b) * a.K + j) * a.dft_stride;
    const int lo = ch * a.chunk_elems;
    const int hi = min(a.V, lo + a.chunk_elems);
    float keep = 0.f, rs = 0.f;
    for (int e = lo + tid; e < hi; e += kMuThreads) {
      const float x = Elem<ES>::load(trow, e);
      const float lp = fmaf(x, a.c, -lp2);
      const float lq = fmaf(Elem<ES>::load(drow, e), a.c, -lq2);
      keep += kept_mass(a.rule, lp, lq, x, thr_row);
      rs += fmaxf(ex2(lp) - ex2(lq), 0.f);
    }
    const float tk = block_sum_fixed(keep, red);
    const float tr = block_sum_fixed(rs, red);
    if (tid == 0) a.mpart[static_cast<int64_t>(blockIdx.x)] = make_float2(tk, tr);
  }
  if (tid == 0) {
    __threadfence();
    const uint32_t ticket = atomicAdd(&a.counters[b], 1u);
    s_last = (ticket == static_cast<uint32_t>(per_req - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last CTA of request b: mu for every emitted draft row j <= min(n, K-1).
  const int jmax = min(n, a.K - 1);
  for (int jj = tid; jj <= jmax; jj += kMuThreads) {
    const float2* pp = a.mpart + (static_cast<int64_t>(b) * a.K + jj) * a.P;
    float keep = 0.f, rsum = 0.f;   // fp32 (FP64 latency is long on this GPU); ~1e-6 relative
    for (int k = 0; k < a.P; ++k) {
      const float2 v = __ldcg(&pp[k]);
      keep += v.x;
      rsum += v.y;
    }
    float lp2, lq2;
    row_lse2<ES>(a, b, jj, lp2, lq2);
    const int64_t o = static_cast<int64_t>(b) * (a.K + 1) + jj;
    const int t = jj < n ? a.drafts[static_cast<int64_t>(b) * a.K + jj] : a.tokens[o];
    if (t < 0 || t >= a.V) continue;
    const float x = Elem<ES>::load(a.tgt + (static_cast<int64_t>(b) * (a.K + 1) + jj) * a.tgt_stride, t);
    const float y = Elem<ES>::load(a.dft + (static_cast<int64_t>(b) * a.K + jj) * a.dft_stride, t);
    const float lp = fmaf(x, a.c, -lp2), lq = fmaf(y, a.c, -lq2);
    const float thr_j = a.rule.thr ? a.rule.thr[static_cast<int64_t>(b) * a.K + jj] : INFINITY;
    const float p = ex2(lp), q = ex2(lq);
    const float res = rsum > 0.f ? fmaxf(p - q, 0.f) / rsum : p;
    const float mu = kept_mass(a.rule, lp, lq, x, thr_j) + (1.f - keep) * res;
    if (a.out_mu) a.out_mu[o] = mu;
  }
  if (tid == 0) a.counters[b] = 0u;
  if (a.fin.out_len) {   // this kernel ends the call
    __syncthreads();
    finish_request(a.fin, fpre, s_stop, b, n, a.K + 1, a.out_tokens, a.out_logprob, a.out_mu, nullptr,
                   a.out_status, s_fin);
  }
}

}  // namespace sv
