// K2: per-request decisions, one CTA per request, launched as a programmatic
// dependent of K1. Everything that depends only on the call's inputs (draft
// tokens, uniforms, the draft tokens' logits, tree links and child lists) is
// read before griddepcontrol.wait, overlapping K1's tail; only K1's row
// statistics are read after it. (K2 can only launch once every K1 CTA has
// passed its own wait on the kernel before the call, so those inputs are
// complete.)
//
// chain_decide_kernel
//   Greedy (mini-sglang PR #134, verify.py): n = first i < K whose draft is
//   out of range or differs from argmax(row i); tokens d_0..d_{n-1}, then
//   argmax(row n).
//   Stochastic (spec-decode README, "How it works"; nanospec README rules):
//   per draft i, a_i = min(1, p(d_i)/q(d_i)) (exact; power ^alpha) or
//   [p(d_i) >= tau] (relaxed), computed in the log2 domain from the row
//   log-sum-exps; accepted iff u_i < a_i; n = first rejection. Row n's draw
//   (residual or bonus) is described for K3.
//   Rows are taken kK2Threads at a time and the first rejection is a block
//   min, so long chains (K+1 = 4096) stop after the block that holds it.
//
// tree_decide_kernel
//   All N rows' statistics and every node's gathered logit (its token in its
//   parent's row) are staged in shared memory; one thread then walks from the
//   root over children in increasing index (nanospec README, tree
//   configuration), with rest kept as a compensated fp32 sum.
#pragma once

#include "finish.cuh"
#include "row_stats.cuh"

namespace sv {

constexpr int kK2Threads = 256;
// Stochastic calls size the decide kernel's registers for three blocks per
// SM, so the draw kernels launched behind it (programmatic dependent launch)
// still find room for their blocks on the SMs that hold a decide block.
// Greedy calls launch nothing behind it and take two blocks per SM, which
// leaves the kernel enough registers not to spill.
constexpr int kK2MinBlocksDraw = 3;
constexpr int kK2MinBlocksGreedy = 2;
// Row-piece slots a decide block stages in shared memory per row set (one
// merged Partial each); a larger range falls back to per-thread merges.
constexpr int kStageSlots = 640;
// Requests whose target plus draft rows number at most kHalfRows are merged
// by one half-warp per row instead (no staging pass).
constexpr int kHalfRows = kK2Threads / 16;
constexpr unsigned long long kEarlyAbortBit = 1ull << 63;   // set in a K1 CTA's byte count
constexpr int kMaxTreeNodes = 1024;

struct RuleArgs {
  int32_t rule;  // 0 exact, 1 relaxed, 2 power
  float tau;
  int32_t top_k;
  float alpha;
  // Relaxed rule with top_k > 0: per tested row, the top_k-th largest logit
  // (topk_threshold_kernel); rank(t) < top_k iff x_t >= it. Else nullptr.
  const float* thr;
};

// Relaxed acceptance of a token with log2 p = lp2 and raw logit x, in a row
// whose rank bound is thr.
__device__ __forceinline__ bool relaxed_accepts(const RuleArgs& r, float lp2, float x, float thr) {
  return ex2(lp2) >= r.tau || (r.top_k > 0 && x >= thr);
}

// Tree acceptance of a child with log2 p = lp2 when `rest` of the parent
// row's mass is left (exact and power rules): min(1, p / rest)^alpha, formed
// in the log2 domain as 2^(alpha * min(0, lp2 - log2 rest)); rest <= 0 (all
// mass removed, by rounding) accepts.
__device__ __forceinline__ float tree_accept(const RuleArgs& r, float lp2, float rest) {
  const float r2 = rest <= 0.f ? 0.f : fminf(0.f, lp2 - lg2(rest));
  return ex2(r.rule == 2 ? r.alpha * r2 : r2);
}

struct ChainArgs {
  const uint8_t* tgt;
  int64_t tgt_stride;    // bytes
  const uint8_t* dft;    // nullptr: deterministic drafts
  int64_t dft_stride;    // bytes
  const int32_t* drafts; // [B, K]
  const float* uniforms; // [B, K+1] (stochastic)
  int32_t B, K, V;
  const Partial* part;   // K1 partials; target rows 0..B*(K+1)-1, then draft rows
  int64_t T;             // K1's flattened element count
  int32_t G;             // K1's CTA count
  float c;               // log2(e) / T (greedy: T = 1)
  int32_t greedy;
  RuleArgs rule;
  int32_t* out_tokens;
  int32_t* out_num;
  float* out_logprob;
  float* out_mu;
  int32_t* out_status;
  DrawDesc* draws;
  int32_t* excl;         // [B * excl_stride]
  int32_t excl_stride;
  uint32_t* mu_counters;    // [B], zeroed here for the mu pass's tickets (or nullptr)
  FinishArgs fin;           // stop / cap / counters (greedy: applied here)
  // Early-exit greedy calls (row_stats_early_kernel): one partial per row at
  // slot `row`; the per-request state is zeroed here for the next call; the
  // K1 CTAs' byte counts are summed into out_bytes.
  int32_t row_partials;
  int32_t* early_state;
  const unsigned long long* cta_bytes;
  int32_t n_cta;
  unsigned long long* out_bytes;
};

// Inputs of one chain position, readable before K1 completes.
struct ChainIn {
  int tok;
  bool bad;
  float u;   // uniform of the accept test (stochastic)
  float x;   // target logit of the draft token (stochastic)
  float y;   // draft logit of the draft token (stochastic, with draft logits)
};

template <int ES>
__device__ __forceinline__ ChainIn load_chain_in(const ChainArgs& a, int b, int i) {
  ChainIn in;
  in.tok = -1;
  in.bad = false;
  in.u = 0.f;
  in.x = -INFINITY;
  in.y = -INFINITY;
  const int R = a.K + 1;
  if (i < a.K) {
    in.tok = a.drafts[static_cast<int64_t>(b) * a.K + i];
    in.bad = in.tok < 0 || in.tok >= a.V;
    if (!a.greedy) {
      in.u = a.uniforms[static_cast<int64_t>(b) * R + i];
      if (!in.bad) {
        in.x = Elem<ES>::load(a.tgt + (static_cast<int64_t>(b) * R + i) * a.tgt_stride, in.tok);
        if (a.dft) in.y = Elem<ES>::load(a.dft + (static_cast<int64_t>(b) * a.K + i) * a.dft_stride, in.tok);
      }
    }
  }
  return in;
}

// (hi, lo) <- (hi + lo) - p as an unevaluated sum: Knuth's TwoSum of hi and -p
// (an error-free addition), with the old low part and the rounding error
// carried in lo.
__device__ __forceinline__ void two_sum_sub(float& hi, float& lo, float p) {
  const float a = hi, b = -p;
  const float s = a + b;
  const float bb = s - a;
  const float err = (a - (s - bb)) + (b - bb);
  const float l = lo + err;
  hi = s + l;
  lo = l - (hi - s);
}

// Rank bound of chain row i (read after the wait: its kernel runs before K2).
__device__ __forceinline__ float row_thr(const ChainArgs& a, int b, int i) {
  return a.rule.thr ? a.rule.thr[static_cast<int64_t>(b) * a.K + i] : INFINITY;
}

// WIDE: the rows span many row-pass CTAs (small batches), so the half-warp
// merge loads four partials per lane per round trip instead of two.
template <int ES, int MIN_BLOCKS, bool WIDE = false>
__global__ void __launch_bounds__(kK2Threads, MIN_BLOCKS) chain_decide_kernel(const ChainArgs a) {
  __shared__ int s_first;
  __shared__ int s_status;
  __shared__ int s_fin[2];
  __shared__ int s_stop[kMaxStopIds];
  __shared__ Partial s_tslots[kStageSlots];   // this block's target rows, one merged Partial per slot
  __shared__ Partial s_dslots[kStageSlots];   // and draft rows
  __shared__ Partial s_rows[kHalfRows];       // short requests: merged target rows, then draft rows
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int K = a.K, R = a.K + 1;
  const float c = a.c;
  const ChainIn pre = load_chain_in<ES>(a, b, tid < R ? tid : R);
  const float u_final = a.greedy ? 0.f : a.uniforms[static_cast<int64_t>(b) * R + K];
  __shared__ FinishPre fpre;   // written by thread 0, read by thread 0 in finish_request
  finish_prefetch(a.fin, b, s_stop, fpre);

  grid_dep_wait();
  grid_dep_launch();

  if (tid == 0) {
    s_status = 0;
    if (a.mu_counters) a.mu_counters[b] = 0;
  }
  if (a.cta_bytes) {   // early-exit call: did any K1 CTA give up waiting?
    __syncthreads();
    bool aborted = false;
    for (int g2 = tid; g2 < a.n_cta; g2 += kK2Threads) aborted |= (a.cta_bytes[g2] & kEarlyAbortBit) != 0;
    if (__syncthreads_or(aborted) && tid == 0) s_status |= SV_STATUS_TIMEOUT;
  }
  int n = -1;
  int base = 0;
  for (; base < R; base += kK2Threads) {
    __syncthreads();   // every thread has read the previous block's s_first
    if (tid == 0) s_first = INT_MAX;
    __syncthreads();
    // Merge this block's rows: a half-warp per row for short requests, else
    // stage the row-piece slots (one merged Partial per slot).
    const int nr = min(kK2Threads, R - base);
    const int nd = min(nr, K - base);   // draft rows of positions base .. base + nd - 1
    const bool with_dft = !a.greedy && a.dft;
    const bool halves = !a.row_partials && base == 0 && R + (with_dft ? K : 0) <= kHalfRows;
    SlotRange tsr, dsr;
    tsr.lo = dsr.lo = 0;
    tsr.n = dsr.n = 0;
    bool tstaged = false, dstaged = false;
    if (halves) {
      const int h = tid >> 4;
      const bool draft_row = h >= R;
      const bool valid = h < R + (with_dft ? K : 0);
      const int64_t row = draft_row ? static_cast<int64_t>(a.B) * R + static_cast<int64_t>(b) * K + (h - R)
                                    : static_cast<int64_t>(b) * R + h;
      float hm, hs;
      int hi, he;
      merge_row_half<WIDE ? 4 : 2>(a.part, row, valid, a.V, a.T, a.G, c, tid & 15, hm, hs, hi, he);
      if (valid && (tid & 15) == 0) {
        Partial o;
        o.m = hm;
        o.s = hs;
        o.idx = hi;
        o.err = he;
        s_rows[h] = o;
      }
      __syncthreads();
    } else if (!a.row_partials) {
      tsr = slot_range(static_cast<int64_t>(b) * R + base, static_cast<int64_t>(b) * R + base + nr - 1, a.V, a.T, a.G);
      tstaged = tsr.n <= kStageSlots;
      if (!a.greedy && a.dft && nd > 0) {
        const int64_t d0 = static_cast<int64_t>(a.B) * R + static_cast<int64_t>(b) * K + base;
        dsr = slot_range(d0, d0 + nd - 1, a.V, a.T, a.G);
        dstaged = dsr.n <= kStageSlots;
      }
      SlotRange none;
      none.lo = 0;
      none.n = 0;
      stage_slots(a.part, tstaged ? tsr : none, s_tslots, dstaged ? dsr : none, s_dslots, c);
      __syncthreads();
    }
    const int i = base + tid;
    const bool active = i < R;
    float m = -INFINITY, s = 0.f, lp2row = 0.f, lq2row = 0.f, lp2 = 0.f, acc = 0.f;
    int idx = INT_MAX, err = 0, st = 0;
    bool zero = false, rej = false;
    const ChainIn in = (base == 0) ? pre : load_chain_in<ES>(a, b, active ? i : R);
    if (active) {
      const int64_t trow = static_cast<int64_t>(b) * R + i;
      const int64_t drow = static_cast<int64_t>(a.B) * R + static_cast<int64_t>(b) * K + i;
      if (a.row_partials || halves) {
        const Partial v = halves ? s_rows[i] : a.part[trow];
        m = v.m;
        s = v.s;
        idx = v.idx;
        err = v.err;
      } else if (tstaged) {
        merge_row_staged(s_tslots, tsr, trow, a.V, a.T, a.G, c, m, s, idx, err);
      } else {
        merge_row_serial(a.part, trow, a.V, a.T, a.G, c, m, s, idx, err);
      }
      lp2row = m * c + log2f(s);
      if (!(fabsf(m) <= FLT_MAX) || !(s > 0.f && s <= FLT_MAX)) st |= SV_STATUS_NONFINITE_ROW;
      if (err) st |= SV_STATUS_TIMEOUT;
      if (i < K) {
        if (a.greedy) {
          rej = in.bad || in.tok != idx;
        } else {
          if (!in.bad) lp2 = in.x * c - lp2row;   // log2 p(t)
          if (a.dft) {
            float md, sd;
            int id, ed;
            if (halves) {
              const Partial v = s_rows[R + i];
              md = v.m;
              sd = v.s;
              id = v.idx;
              ed = v.err;
            } else if (dstaged) {
              merge_row_staged(s_dslots, dsr, drow, a.V, a.T, a.G, c, md, sd, id, ed);
            } else {
              merge_row_serial(a.part, drow, a.V, a.T, a.G, c, md, sd, id, ed);
            }
            lq2row = md * c + log2f(sd);
            if (!(fabsf(md) <= FLT_MAX) || !(sd > 0.f && sd <= FLT_MAX)) st |= SV_STATUS_NONFINITE_ROW;
            if (ed) st |= SV_STATUS_TIMEOUT;
            if (!in.bad) {
              const float lq2 = in.y * c - lq2row;
              if (lp2 == -INFINITY && lq2 == -INFINITY) {
                zero = true;
              } else {
                const float r2 = fminf(0.f, lp2 - lq2);   // log2 min(1, p/q)
                if (a.rule.rule == 1) acc = relaxed_accepts(a.rule, lp2, in.x, row_thr(a, b, i)) ? 1.f : 0.f;
                else if (a.rule.rule == 2) acc = ex2(a.rule.alpha * r2);
                else acc = ex2(r2);
              }
            }
          } else if (!in.bad) {   // deterministic draft, rest_1 = 1
            const float r2 = fminf(0.f, lp2);
            if (a.rule.rule == 1) acc = relaxed_accepts(a.rule, lp2, in.x, row_thr(a, b, i)) ? 1.f : 0.f;
            else if (a.rule.rule == 2) acc = ex2(a.rule.alpha * r2);
            else acc = ex2(r2);
          }
          rej = in.bad || zero || !(in.u < acc);
        }
      }
      if (rej) atomicMin(&s_first, i);
    }
    __syncthreads();
    const int first = s_first;
    const bool last_block = base + kK2Threads >= R;
    const int nb = first != INT_MAX ? first : (last_block ? K : INT_MAX);
    if (active) {
      const int64_t o = static_cast<int64_t>(b) * R + i;
      if (i <= nb) {
        int stat = st;
        if (i == nb && i < K) {
          if (in.bad) stat |= SV_STATUS_BAD_TOKEN;
          if (zero) stat |= SV_STATUS_ZERO_MASS;
        }
        if (stat) atomicOr(&s_status, stat);
      }
      if (a.greedy) {
        int out_tok = -1;
        float lp = 0.f, mu = 0.f;
        if (i <= nb) {
          out_tok = (i < nb) ? in.tok : idx;
          lp = -log2f(s) * kLn2;   // emitted tokens are argmaxes, so x[tok] = m
          mu = 1.f;
        }
        a.out_tokens[o] = out_tok;
        if (a.out_logprob) a.out_logprob[o] = lp;
        if (a.out_mu) a.out_mu[o] = mu;
      } else {
        if (i < nb) {
          a.out_tokens[o] = in.tok;
          if (a.out_logprob) a.out_logprob[o] = lp2 * kLn2;
          if (a.out_mu) a.out_mu[o] = a.dft ? ex2(lp2) : acc;
        } else if (i == nb) {
          DrawDesc d;
          d.pos = i;
          d.u = u_final;
          d.t_row = static_cast<int32_t>(static_cast<int64_t>(b) * R + i);
          d.d_row = static_cast<int32_t>(static_cast<int64_t>(b) * K + i);
          d.lp2 = lp2row;
          d.lq2 = lq2row;
          d.scale = 1.f;
          d.n_excl = 0;
          d.pad0 = d.pad1 = d.pad2 = 0;
          if (i == K) {
            d.type = kDrawP;
          } else if (a.dft) {
            d.type = kDrawResid;
          } else {
            d.type = kDrawMaskedP;
            d.scale = 1.f - acc;
            if (!in.bad) {
              a.excl[static_cast<int64_t>(b) * a.excl_stride] = in.tok;
              d.n_excl = 1;
            }
          }
          a.draws[b] = d;
          // K3 writes this position's token, log-prob and mu.
        } else {
          a.out_tokens[o] = -1;
          if (a.out_logprob) a.out_logprob[o] = 0.f;
          if (a.out_mu) a.out_mu[o] = 0.f;
        }
      }
    }
    if (nb != INT_MAX) {
      n = nb;
      break;
    }
  }
  // Columns after the block that held the decision.
  for (int j = base + kK2Threads + tid; j < R; j += kK2Threads) {
    const int64_t o = static_cast<int64_t>(b) * R + j;
    a.out_tokens[o] = -1;
    if (a.out_logprob) a.out_logprob[o] = 0.f;
    if (a.out_mu) a.out_mu[o] = 0.f;
  }
  __syncthreads();
  if (tid == 0) {
    a.out_num[b] = n;
    if (a.out_status) a.out_status[b] = s_status;
    if (a.early_state) {   // ready for the next call: mismatch word and finished-row count
      a.early_state[b] = 0;
      a.early_state[a.B + b] = 0;
    }
  }
  if (a.out_bytes && b == 0) {   // bytes the early-exit K1 read: per-thread, warp, then block sums
    __shared__ unsigned long long s_bytes[kK2Threads / 32];
    unsigned long long t = 0;
    for (int g2 = tid; g2 < a.n_cta; g2 += kK2Threads) t += a.cta_bytes[g2] & ~kEarlyAbortBit;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if ((tid & 31) == 0) s_bytes[tid >> 5] = t;
    __syncthreads();
    if (tid == 0) {
      unsigned long long tot = 0;
#pragma unroll
      for (int k = 0; k < kK2Threads / 32; ++k) tot += s_bytes[k];
      a.out_bytes[0] = tot;
    }
  }
  if (a.greedy && a.fin.out_len) {   // greedy: this kernel ends the call
    __syncthreads();
    finish_request(a.fin, fpre, s_stop, b, n, R, a.out_tokens, a.out_logprob, a.out_mu, nullptr, a.out_status,
                   s_fin);
  }
}

struct TreeArgs {
  const uint8_t* tgt;
  int64_t tgt_stride;      // bytes
  const int32_t* tokens;   // [B, N]
  const int32_t* parents;  // [B, N]
  const float* uniforms;   // [B, N] (stochastic)
  int32_t B, N, V, max_depth;
  const Partial* part;     // K1 partials of the B*N rows
  int64_t T;
  int32_t G;
  float c;                 // log2(e) / T (greedy: T = 1)
  int32_t greedy;
  RuleArgs rule;
  int32_t* out_tokens;     // [B, W], W = max_depth + 1
  int32_t* out_nodes;
  int32_t* out_num;
  float* out_logprob;
  float* out_mu;
  int32_t* out_status;
  DrawDesc* draws;
  int32_t* excl;
  int32_t excl_stride;
  FinishArgs fin;          // stop / cap / counters (greedy walk: applied here)
};

template <int ES>
__global__ void __launch_bounds__(kK2Threads) tree_decide_kernel(const TreeArgs a) {
  __shared__ float sm_m[kMaxTreeNodes];     // row max
  __shared__ float sm_l2[kMaxTreeNodes];    // row lse, log2 domain
  __shared__ float sm_g[kMaxTreeNodes];     // node token's logit in its parent's row
  __shared__ float sm_u[kMaxTreeNodes];     // node's uniform
  __shared__ int sm_am[kMaxTreeNodes];      // row argmax
  __shared__ int sm_tok[kMaxTreeNodes];
  __shared__ int sm_par[kMaxTreeNodes];     // -1 for the root and bad links
  __shared__ int sm_first[kMaxTreeNodes];   // first child
  __shared__ int sm_next[kMaxTreeNodes];    // next sibling
  __shared__ unsigned char sm_bad[kMaxTreeNodes];  // row not finite / timed out
  __shared__ int s_status;
  __shared__ int s_n, s_fin[2];
  __shared__ int s_stop[kMaxStopIds];
  __shared__ Partial s_slots[kStageSlots];  // the request's row-piece slots, one merged Partial each

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int N = a.N, W = a.max_depth + 1;
  const float c = a.c;

  // Call inputs: links, tokens, uniforms and the gathered logits.
  if (tid == 0) s_status = 0;
  __syncthreads();
  for (int n = tid; n < N; n += kK2Threads) {
    const int64_t row = static_cast<int64_t>(b) * N + n;
    const int par = a.parents[row];
    const int tok = a.tokens[row];
    const bool link_ok = (n == 0) ? (par == -1) : (par >= 0 && par < n);
    if (!link_ok) atomicOr(&s_status, SV_STATUS_BAD_PARENT);
    const int p = (n > 0 && link_ok) ? par : -1;
    sm_par[n] = p;
    sm_tok[n] = tok;
    sm_u[n] = a.greedy ? 0.f : a.uniforms[row];
    float gl = -INFINITY;
    if (p >= 0 && tok >= 0 && tok < a.V)
      gl = Elem<ES>::load(a.tgt + (static_cast<int64_t>(b) * N + p) * a.tgt_stride, tok);
    sm_g[n] = gl;
    sm_first[n] = -1;
  }
  __syncthreads();
  __shared__ FinishPre fpre;   // written by thread 0, read by thread 0 in finish_request
  finish_prefetch(a.fin, b, s_stop, fpre);
  if (tid == 0) {
    for (int n = N - 1; n >= 1; --n) {   // reverse insertion: lists in increasing index
      const int p = sm_par[n];
      if (p >= 0) {
        sm_next[n] = sm_first[p];
        sm_first[p] = n;
      }
    }
  }

  grid_dep_wait();
  grid_dep_launch();

  const SlotRange sr = slot_range(static_cast<int64_t>(b) * N, static_cast<int64_t>(b) * N + N - 1, a.V, a.T, a.G);
  const bool staged = sr.n <= kStageSlots;
  if (staged) {
    SlotRange none;
    none.lo = 0;
    none.n = 0;
    stage_slots(a.part, sr, s_slots, none, nullptr, c);
    __syncthreads();
  }
  for (int n = tid; n < N; n += kK2Threads) {
    float m, s;
    int idx, err;
    if (staged) merge_row_staged(s_slots, sr, static_cast<int64_t>(b) * N + n, a.V, a.T, a.G, c, m, s, idx, err);
    else merge_row_serial(a.part, static_cast<int64_t>(b) * N + n, a.V, a.T, a.G, c, m, s, idx, err);
    sm_m[n] = m;
    sm_l2[n] = m * c + log2f(s);
    sm_am[n] = idx;
    sm_bad[n] = static_cast<unsigned char>(
        ((!(fabsf(m) <= FLT_MAX) || !(s > 0.f && s <= FLT_MAX)) ? SV_STATUS_NONFINITE_ROW : 0) |
        (err ? SV_STATUS_TIMEOUT : 0));
  }
  __syncthreads();
  if (tid == 0) {
    int status = 0;
    int cur = 0, depth = 0;
    const int64_t ob = static_cast<int64_t>(b) * W;
    int32_t* excl = a.excl + static_cast<int64_t>(b) * a.excl_stride;
    while (true) {
      a.out_nodes[ob + depth] = cur;
      status |= sm_bad[cur];
      int kid = sm_first[cur];
      if (depth == a.max_depth && kid >= 0) {
        status |= SV_STATUS_DEPTH_EXCEEDED;
        kid = -1;
      }
      if (a.greedy) {
        const int am = sm_am[cur];
        int nxt = -1;
        for (; kid >= 0; kid = sm_next[kid]) {
          const int t = sm_tok[kid];
          if (t < 0 || t >= a.V) {
            status |= SV_STATUS_BAD_TOKEN;
            continue;
          }
          if (t == am) {
            nxt = kid;
            break;
          }
        }
        a.out_tokens[ob + depth] = am;
        if (a.out_logprob) a.out_logprob[ob + depth] = (sm_m[cur] * c - sm_l2[cur]) * kLn2;
        if (a.out_mu) a.out_mu[ob + depth] = 1.f;
        if (nxt < 0) break;
        cur = nxt;
        ++depth;
        continue;
      }
      // rest = 1 - (rejected mass) as an unevaluated fp32 sum rest_hi + rest_lo
      // (TwoSum keeps it exact to ~1e-14 when the rejected mass nears 1; FP64
      // latency on this GPU made a double walk several microseconds long)
      float rest_hi = 1.f, rest_lo = 0.f, reach = 1.f;
      int nrej = 0, accepted = -1;
      for (; kid >= 0; kid = sm_next[kid]) {
        const int t = sm_tok[kid];
        float acc = 0.f;
        float lp2 = -INFINITY;
        bool counted = false;
        if (t < 0 || t >= a.V) {
          status |= SV_STATUS_BAD_TOKEN;
        } else {
          bool dup = false;
          for (int r = 0; r < nrej; ++r) dup |= (excl[r] == t);
          if (!dup) {
            counted = true;
            lp2 = sm_g[kid] * c - sm_l2[cur];
            const float p = ex2(lp2);
            if (a.rule.rule == 1) {
              const float thr = a.rule.thr ? a.rule.thr[static_cast<int64_t>(b) * N + cur] : INFINITY;
              acc = relaxed_accepts(a.rule, lp2, sm_g[kid], thr) ? 1.f : 0.f;
            } else {
              acc = tree_accept(a.rule, lp2, rest_hi + rest_lo);
            }
            two_sum_sub(rest_hi, rest_lo, p);
          }
        }
        if (sm_u[kid] < acc) {
          accepted = kid;
          a.out_tokens[ob + depth] = t;
          if (a.out_logprob) a.out_logprob[ob + depth] = lp2 * kLn2;
          if (a.out_mu) a.out_mu[ob + depth] = reach * acc;
          break;
        }
        reach *= (1.f - acc);
        if (counted) excl[nrej++] = t;
      }
      if (accepted >= 0) {
        cur = accepted;
        ++depth;
        continue;
      }
      DrawDesc d;
      d.type = nrej > 0 ? kDrawMaskedP : kDrawP;
      d.t_row = static_cast<int32_t>(static_cast<int64_t>(b) * N + cur);
      d.d_row = 0;
      d.pos = depth;
      d.u = sm_u[0];
      d.lp2 = sm_l2[cur];
      d.lq2 = 0.f;
      d.scale = reach;
      d.n_excl = nrej;
      d.pad0 = d.pad1 = d.pad2 = 0;
      a.draws[b] = d;
      break;
    }
    a.out_num[b] = depth;
    s_n = depth;
    for (int j = depth + 1; j < W; ++j) {
      a.out_tokens[ob + j] = -1;
      a.out_nodes[ob + j] = -1;
      if (a.out_logprob) a.out_logprob[ob + j] = 0.f;
      if (a.out_mu) a.out_mu[ob + j] = 0.f;
    }
    atomicOr(&s_status, status);
  }
  __syncthreads();
  if (tid == 0 && a.out_status) a.out_status[b] = s_status;
  if (a.greedy && a.fin.out_len) {   // greedy walk: this kernel ends the call
    __syncthreads();
    finish_request(a.fin, fpre, s_stop, b, s_n, W, a.out_tokens, a.out_logprob, a.out_mu, a.out_nodes,
                   a.out_status, s_fin);
  }
}

}  // namespace sv
