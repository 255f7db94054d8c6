// The step after a verify decision: stop-set and max-new-tokens truncation
// and per-request counters, done by whichever kernel finishes a request
// (mini-sglang PR #134: Known limitations, multi-token stop sets; engine.py,
// accept_length and accept_rate counters; spec-decode README CLI: tokens per
// target pass and acceptance rate).
//
// A call emits tokens[0..n]. The request stops at the first emitted token in
// the stop set (kept), max_new[b] caps the tokens kept (clamped at 0), and
// positions kept..n are cleared (token -1, log-prob 0, mu 0, node -1).
// Status gains STOPPED (64) when a stop token is kept and CAPPED (128) when
// the cap removed an emitted token. counters[b] accumulate (rounds, drafts
// offered, drafts accepted by the rule, tokens kept).
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kStatusStopped = SV_STATUS_STOPPED;
constexpr int kStatusCapped = SV_STATUS_CAPPED;
constexpr int kMaxStopIds = 16;

struct FinishArgs {
  const int32_t* stop_ids;   // [n_stop]
  int32_t n_stop;
  const int32_t* max_new;    // [B] or nullptr
  int32_t* out_len;          // [B]; nullptr: no finish step in this call
  long long* counters;       // [B, 4] or nullptr
  int32_t offered;           // drafts offered per call: K (chain) or max_depth (tree)
};

// The finish step's inputs for request b, read at kernel start (before the
// dependency wait: they are call inputs, and only this step writes the
// counters, once per call at its end). Stop ids go to shared memory; thread 0
// writes the cap and the counters into `pre`, which the kernels keep in
// shared memory (so no thread holds them in registers for the whole kernel).
struct FinishPre {
  int cap;            // INT_MAX when there is no cap
  long long c[4];
};

__device__ __forceinline__ void finish_prefetch(const FinishArgs& f, int b, int* s_stop, FinishPre& pre) {
  if (!f.out_len) return;
  if (static_cast<int>(threadIdx.x) < f.n_stop) s_stop[threadIdx.x] = __ldg(f.stop_ids + threadIdx.x);
  if (threadIdx.x == 0) {
    pre.cap = f.max_new ? max(0, __ldg(f.max_new + b)) : INT_MAX;
#pragma unroll
    for (int k = 0; k < 4; ++k) pre.c[k] = f.counters ? f.counters[static_cast<int64_t>(b) * 4 + k] : 0;
  }
}

// Block-cooperative: every thread of the CTA calls it once the request's
// outputs (row b of `cols` columns) are final and visible to the block, after
// finish_prefetch in the same kernel.
__device__ __forceinline__ void finish_request(const FinishArgs& f, const FinishPre& pre, const int* s_stop,
                                               int b, int n, int cols, int32_t* tokens, float* logprob,
                                               float* mu, int32_t* nodes, int32_t* status, int* s_first) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int64_t rb = static_cast<int64_t>(b) * cols;
  if (tid == 0) *s_first = INT_MAX;
  __syncthreads();
  for (int j = tid; j <= n; j += nt) {
    const int t = tokens[rb + j];
    for (int k = 0; k < f.n_stop; ++k) {
      if (t == s_stop[k]) {
        atomicMin(s_first, j);
        break;
      }
    }
  }
  __syncthreads();
  const int first = *s_first;
  int kept = n + 1;
  if (first != INT_MAX) kept = first + 1;
  if (tid == 0) {   // thread 0 applies the cap and broadcasts the kept count
    bool stopped = first != INT_MAX, capped = false;
    if (pre.cap < kept) {
      kept = pre.cap;
      capped = true;
      stopped = false;   // a stop token at index >= cap was cut off
    }
    s_first[1] = kept;
    f.out_len[b] = kept;
    if (status) status[b] |= (stopped ? kStatusStopped : 0) | (capped ? kStatusCapped : 0);
    if (f.counters) {
      long long* c = f.counters + static_cast<int64_t>(b) * 4;
      c[0] = pre.c[0] + 1;
      c[1] = pre.c[1] + f.offered;
      c[2] = pre.c[2] + n;
      c[3] = pre.c[3] + kept;
    }
  }
  __syncthreads();
  kept = s_first[1];
  for (int j = kept + tid; j <= n; j += nt) {
    tokens[rb + j] = -1;
    if (logprob) logprob[rb + j] = 0.f;
    if (mu) mu[rb + j] = 0.f;
    if (nodes) nodes[rb + j] = -1;
  }
}

}  // namespace sv
