// Stochastic tree verification in one kernel: the row-statistics merge, the
// walk (nanospec README, tree configuration) and the draw that ends it (the
// masked or bonus sample; spec-decode README, "How it works" for the inverse
// CDF), for one request per thread-block cluster.
//
// The same computation as tree_decide_kernel followed by draw_sum_kernel and
// draw_pick_kernel, without their two kernel boundaries and global round
// trips. A cluster of kTwCluster CTAs serves request b:
//
//  1. CTA 0 merges the K1 partials of the request's N rows (the decide
//     kernel's staged merge, so the statistics are the same bits), forms
//     every node's log2 p in parallel, and one thread walks from the root as
//     the decide kernel does (same arithmetic and order), writing the
//     accepted path. The draw descriptor and the rejected tokens are stored
//     into every CTA's shared memory (distributed shared memory).
//  2. Cluster barrier 1. CTA r copies chunks [r * nch, (r + 1) * nch) of the
//     drawn row (kK3ChunkBytes each, 1-D bulk copies) into its shared memory,
//     masks the rejected tokens and the row's end with -inf, sums the weights
//     per 16-byte vector and per chunk, and stores the chunk sums into every
//     CTA's shared memory.
//  3. Cluster barrier 2. Every CTA finds the chunk where u * S falls (warp
//     scans over the chunk sums); the CTA holding that chunk scans its
//     vector sums, resolves the token inside the crossing vector, and
//     writes the draw, the status and the finish step.
//
// After barrier 2 no CTA touches another's shared memory, so the CTAs not
// holding the drawn chunk simply exit. (Barrier 0, every CTA of the cluster
// running, precedes the first remote store.) The copies wait on an mbarrier
// with the bounded wait; a wait that gives up makes the chunk sums NaN, and
// the request reports SV_STATUS_TIMEOUT. Requires 16-byte-aligned rows (the
// base and the row stride) so each chunk starts on a 16-byte boundary; the
// host uses the three-kernel path otherwise.
#pragma once

#include "decide.cuh"
#include "draw.cuh"
#include "finish.cuh"

namespace sv {

constexpr int kTwCluster = 8;                 // CTAs per request
constexpr int kTwThreads = 256;
constexpr int kTwWarps = kTwThreads / 32;
constexpr int kTwMaxChunks = 6;               // chunks of the drawn row one CTA holds
constexpr int kTwMaxP = kTwCluster * kTwMaxChunks;
constexpr int kTwVecs = kK3ChunkBytes / 16;   // 16-byte vectors per chunk
constexpr int kTwVecsPerThread = kTwVecs / kTwThreads;
static_assert(kTwVecsPerThread * kTwThreads == kTwVecs, "whole vectors per thread");

// The walk's result, as CTA 0 hands it to the cluster.
struct TwDraw {
  int32_t type;     // DrawType
  int32_t t_row;    // global target row
  int32_t pos;      // output column
  int32_t n_excl;   // rejected tokens (masked draw)
  int32_t status;   // the walk's status bits
  float u, lp2, scale;
};
static_assert(sizeof(TwDraw) == 32, "eight 32-bit words");

struct TwArgs {
  TreeArgs t;          // tree inputs, outputs, K1 partials, rule, finish step
  uintptr_t tgt_hi;    // end of the target buffer (bytes)
  int32_t P;           // chunks per row
  int32_t chunk_elems;
  int32_t nch;         // chunks per CTA: ceil(P / kTwCluster)
};

// ------------------------------------------------ cluster / distributed shared memory

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_cluster(uint32_t addr, float v) { st_cluster(addr, __float_as_uint(v)); }

__device__ __forceinline__ void st_cluster(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}

// Cluster-wide barrier: every thread of every CTA arrives (release: its
// earlier stores, shared and global, become visible to the waiters) and
// waits (acquire).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// Dynamic shared-memory layout for N nodes and nch chunks per CTA (the host
// sizes the launch with the same function).
struct TwLayout {
  uint32_t l2, g, u, lp, p, racc, xp, tok, par, first, next, dup, bad, excl, slots, vsum, chunks, total;
};

__host__ __device__ constexpr uint32_t tw_align(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline TwLayout tw_layout(int N, int nch) {
  TwLayout L{};
  const uint32_t n4 = tw_align(static_cast<uint32_t>(N), 4) * 4u;   // one 32-bit word per node
  uint32_t o = 0;
  L.l2 = o;    o += n4;
  L.g = o;     o += n4;
  L.u = o;     o += n4;
  L.lp = o;    o += n4;
  L.p = o;     o += n4;
  L.racc = o;  o += n4;
  L.xp = o;    o += n4;
  L.tok = o;   o += n4;
  L.par = o;   o += n4;
  L.first = o; o += n4;
  L.next = o;  o += n4;
  L.dup = o;   o += n4;
  L.bad = o;   o += n4;
  L.excl = o;  o += n4;
  o = tw_align(o, 16);
  L.slots = o; o += static_cast<uint32_t>(kStageSlots * sizeof(Partial));
  L.vsum = o;  o += static_cast<uint32_t>(nch) * kTwVecs * 4u;   // weight sum of each 16-byte vector
  o = tw_align(o, 128);
  L.chunks = o; o += static_cast<uint32_t>(nch) * kK3ChunkBytes;
  L.total = o;
  return L;
}

template <int ES>
__global__ void __cluster_dims__(kTwCluster, 1, 1) __launch_bounds__(kTwThreads, 1)
    tree_walk_draw_kernel(const TwArgs w) {
  constexpr int NV = Elem<ES>::kVec;   // elements per 16-byte vector
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t s_bar;           // the chunk copies
  __shared__ TwDraw s_draw;                          // CTA 0 stores it into every CTA
  __shared__ float2 s_csum[kTwMaxP];                 // (sum w, sum p) per chunk, in every CTA
  __shared__ float s_red[kTwMaxChunks][kTwWarps];    // warp sums of w per local chunk
  __shared__ float s_wsum[kTwWarps];                 // the owner's block scan: warp totals
  __shared__ int s_stop[kMaxStopIds];
  __shared__ FinishPre fpre;
  __shared__ int s_fin[2];
  __shared__ int s_cand[kTwWarps];                   // first crossing thread per warp
  __shared__ int s_wlast[kTwWarps];                  // last thread with weight per warp
  __shared__ int s_err, s_chunk, s_usep, s_link;
  __shared__ float s_thr, s_S;

  const TreeArgs& a = w.t;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int b = static_cast<int>(blockIdx.x) / kTwCluster;
  const int N = a.N, W = a.max_depth + 1;
  const float c = a.c;
  const TwLayout L = tw_layout(N, w.nch);
  float* sm_l2 = reinterpret_cast<float*>(smem + L.l2);     // row lse, log2 domain
  float* sm_g = reinterpret_cast<float*>(smem + L.g);       // node token's logit in its parent's row
  float* sm_u = reinterpret_cast<float*>(smem + L.u);       // node's uniform
  float* sm_lp = reinterpret_cast<float*>(smem + L.lp);     // node token's log2 p in its parent's row
  float* sm_p = reinterpret_cast<float*>(smem + L.p);       // 2^lp
  float* sm_racc = reinterpret_cast<float*>(smem + L.racc); // relaxed rule: the node's acceptance (0 / 1)
  float* sm_xp = reinterpret_cast<float*>(smem + L.xp);     // p of each rejected token (draw masking)
  int* sm_tok = reinterpret_cast<int*>(smem + L.tok);
  int* sm_par = reinterpret_cast<int*>(smem + L.par);       // -1 for the root and bad links
  int* sm_first = reinterpret_cast<int*>(smem + L.first);   // first child
  int* sm_next = reinterpret_cast<int*>(smem + L.next);     // next sibling
  int* sm_dup = reinterpret_cast<int*>(smem + L.dup);       // an earlier sibling offers the same token
  int* sm_bad = reinterpret_cast<int*>(smem + L.bad);       // row not finite / timed out
  int* s_excl = reinterpret_cast<int*>(smem + L.excl);      // rejected tokens of the draw's node
  Partial* s_slots = reinterpret_cast<Partial*>(smem + L.slots);
  float* s_vsum = reinterpret_cast<float*>(smem + L.vsum);   // [nch][kTwVecs]
  uint8_t* chunks = smem + L.chunks;

  cluster_arrive_relaxed();   // barrier 0: this CTA has started (awaited before any remote store)
  if (tid == 0) {
    s_err = 0;
    s_link = 0;
    mbar_init(smem_u32(&s_bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Call inputs (CTA 0 walks): links, tokens, uniforms and the gathered logits.
  if (rank == 0) {
    for (int n = tid; n < N; n += kTwThreads) {
      const int64_t row = static_cast<int64_t>(b) * N + n;
      const int par = a.parents[row];
      const int tok = a.tokens[row];
      const bool link_ok = (n == 0) ? (par == -1) : (par >= 0 && par < n);
      if (!link_ok) atomicOr(&s_link, SV_STATUS_BAD_PARENT);
      const int p = (n > 0 && link_ok) ? par : -1;
      sm_par[n] = p;
      sm_tok[n] = tok;
      sm_u[n] = a.uniforms[row];
      float gl = -INFINITY;
      if (p >= 0 && tok >= 0 && tok < a.V)
        gl = Elem<ES>::load(a.tgt + (static_cast<int64_t>(b) * N + p) * a.tgt_stride, tok);
      sm_g[n] = gl;
      sm_first[n] = -1;
    }
  }
  finish_prefetch(a.fin, b, s_stop, fpre);
  __syncthreads();
  if (rank == 0) {
    if (tid == 0) {
      for (int n = N - 1; n >= 1; --n) {   // reverse insertion: lists in increasing index
        const int p = sm_par[n];
        if (p >= 0) {
          sm_next[n] = sm_first[p];
          sm_first[p] = n;
        }
      }
    }
    __syncthreads();
    // A child whose in-range token an earlier sibling already offered is not
    // tested again (its token was removed from the parent's row).
    for (int n = tid; n < N; n += kTwThreads) {
      const int t = sm_tok[n], p = sm_par[n];
      int dup = 0;
      if (p >= 0 && t >= 0 && t < a.V)
        for (int m = sm_first[p]; m >= 0 && m != n; m = sm_next[m]) dup |= sm_tok[m] == t;
      sm_dup[n] = dup;
    }
  }

  grid_dep_wait();
  grid_dep_launch();

  cluster_wait();   // barrier 0: every CTA of the cluster runs (before any remote store)
  const int64_t rb = static_cast<int64_t>(b) * N;

  // ---- 1. CTA 0: the rows' statistics (the decide kernel's staged merge;
  // the merge is one L2 round trip however many rows a CTA takes)
  if (rank == 0) {
    const SlotRange sr = slot_range(rb, rb + N - 1, a.V, a.T, a.G);
    const bool staged = sr.n <= kStageSlots;
    if (staged) {
      SlotRange none;
      none.lo = 0;
      none.n = 0;
      stage_slots(a.part, sr, s_slots, none, nullptr, c);
      __syncthreads();
    }
    for (int n = tid; n < N; n += kTwThreads) {
      float m, s;
      int idx, err;
      if (staged) merge_row_staged(s_slots, sr, rb + n, a.V, a.T, a.G, c, m, s, idx, err);
      else merge_row_serial(a.part, rb + n, a.V, a.T, a.G, c, m, s, idx, err);
      sm_l2[n] = m * c + log2f(s);
      sm_bad[n] = ((!(fabsf(m) <= FLT_MAX) || !(s > 0.f && s <= FLT_MAX)) ? SV_STATUS_NONFINITE_ROW : 0) |
                  (err ? SV_STATUS_TIMEOUT : 0);
    }
    __syncthreads();
  }

  // ---- 2. CTA 0: every node's log2 p (and relaxed acceptance), then the walk
  if (rank == 0) {
    for (int n = tid; n < N; n += kTwThreads) {
      const int p = sm_par[n];
      const float lp2 = p >= 0 ? sm_g[n] * c - sm_l2[p] : -INFINITY;
      sm_lp[n] = lp2;
      sm_p[n] = ex2(lp2);
      if (a.rule.rule == 1 && p >= 0) {
        const float thr = a.rule.thr ? a.rule.thr[rb + p] : INFINITY;
        sm_racc[n] = relaxed_accepts(a.rule, lp2, sm_g[n], thr) ? 1.f : 0.f;
      }
    }
    __syncthreads();
    if (tid == 0) {
      int status = s_link;
      int cur = 0, depth = 0;
      const int64_t ob = static_cast<int64_t>(b) * W;
      TwDraw d;
      while (true) {
        a.out_nodes[ob + depth] = cur;
        status |= sm_bad[cur];
        int kid = sm_first[cur];
        if (depth == a.max_depth && kid >= 0) {
          status |= SV_STATUS_DEPTH_EXCEEDED;
          kid = -1;
        }
        // rest = 1 - (rejected mass) as an unevaluated fp32 sum rest_hi + rest_lo
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
            if (!sm_dup[kid]) {
              counted = true;
              lp2 = sm_lp[kid];
              acc = a.rule.rule == 1 ? sm_racc[kid] : tree_accept(a.rule, lp2, rest_hi + rest_lo);
              two_sum_sub(rest_hi, rest_lo, sm_p[kid]);
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
          if (counted) s_excl[nrej++] = t;
        }
        if (accepted >= 0) {
          cur = accepted;
          ++depth;
          continue;
        }
        d.type = nrej > 0 ? kDrawMaskedP : kDrawP;
        d.t_row = static_cast<int32_t>(rb + cur);
        d.pos = depth;
        d.n_excl = nrej;
        d.u = sm_u[0];
        d.lp2 = sm_l2[cur];
        d.scale = reach;
        break;
      }
      a.out_num[b] = depth;
      for (int j = depth + 1; j < W; ++j) {
        a.out_tokens[ob + j] = -1;
        a.out_nodes[ob + j] = -1;
        if (a.out_logprob) a.out_logprob[ob + j] = 0.f;
        if (a.out_mu) a.out_mu[ob + j] = 0.f;
      }
      d.status = status;
      s_draw = d;
    }
    __syncthreads();
    // The draw and the rejected tokens into the other CTAs.
    const int nw = 8 + s_draw.n_excl;
    const uint32_t* dw = reinterpret_cast<const uint32_t*>(&s_draw);
    for (int q = tid; q < (kTwCluster - 1) * nw; q += kTwThreads) {
      const int dst = 1 + q / nw, k = q - (q / nw) * nw;
      if (k < 8) st_cluster(map_rank(smem_u32(dw + k), dst), dw[k]);
      else st_cluster(map_rank(smem_u32(s_excl + (k - 8)), dst), static_cast<uint32_t>(s_excl[k - 8]));
    }
  }
  cluster_sync();   // barrier 1: every CTA holds the draw

  // ---- 3. this CTA's chunks of the drawn row: copy, mask, sum
  const TwDraw d = s_draw;
  const int ce = w.chunk_elems;
  const int k0 = static_cast<int>(rank) * w.nch;
  const int nloc = max(0, min(w.P, k0 + w.nch) - k0);
  const uint8_t* trow = a.tgt + static_cast<int64_t>(d.t_row) * a.tgt_stride;
  // Bytes copied for local chunk ci: the chunk rounded up to whole vectors,
  // cut back to whole vectors inside the buffer at its very end.
  auto copy_bytes = [&](int ci) -> uint32_t {
    const int lo = (k0 + ci) * ce, hi = min(a.V, lo + ce);
    const uintptr_t src = reinterpret_cast<uintptr_t>(trow) + static_cast<uintptr_t>(lo) * ES;
    uint32_t nb = static_cast<uint32_t>(((hi - lo) * ES + 15) & ~15);
    if (src + nb > w.tgt_hi) nb = static_cast<uint32_t>((w.tgt_hi - src) & ~static_cast<uintptr_t>(15));
    return nb;
  };
  if (tid == 0) {
    uint32_t total = 0;
    for (int ci = 0; ci < nloc; ++ci) total += copy_bytes(ci);
    const uint32_t bar = smem_u32(&s_bar);
    mbar_arrive_expect_tx(bar, total);
    for (int ci = 0; ci < nloc; ++ci) {
      const uint32_t nb = copy_bytes(ci);
      if (nb) bulk_g2s(smem_u32(chunks + ci * kK3ChunkBytes), trow + static_cast<int64_t>(k0 + ci) * ce * ES, nb, bar);
    }
  }
  if (!mbar_wait_bounded(smem_u32(&s_bar), 0)) atomicOr(&s_err, 1);
  // Elements a cut-back copy left out (from global memory), and -inf past the
  // row's end up to the vector boundary (a full copy brought the next row's
  // first elements or the stride's padding there).
  for (int ci = 0; ci < nloc; ++ci) {
    const int lo = (k0 + ci) * ce, hi = min(a.V, lo + ce);
    const int got = static_cast<int>(copy_bytes(ci)) / ES;
    const int vend = (hi - lo + NV - 1) / NV * NV;
    const int j = min(got, hi - lo) + tid;
    if (j < vend) {
      uint8_t* e = chunks + ci * kK3ChunkBytes + j * ES;
      if constexpr (ES == 4) {
        *reinterpret_cast<float*>(e) = lo + j < hi ? Elem<4>::load(trow, lo + j) : -INFINITY;
      } else {
        *reinterpret_cast<unsigned short*>(e) =
            lo + j < hi ? __ldg(reinterpret_cast<const unsigned short*>(trow) + lo + j) : static_cast<unsigned short>(0xff80u);
      }
    }
  }
  __syncthreads();
  // Rejected tokens: their p (for the unmasked sums), then -inf in the copy.
  const int nex = d.type == kDrawMaskedP ? d.n_excl : 0;
  const int lo_cta = k0 * ce, hi_cta = min(a.V, (k0 + nloc) * ce);
  for (int e = tid; e < nex; e += kTwThreads) {
    const int t = s_excl[e];
    float xp = 0.f;
    if (t >= lo_cta && t < hi_cta) {
      uint8_t* el = chunks + ((t - lo_cta) / ce) * kK3ChunkBytes + ((t - lo_cta) % ce) * ES;
      float x;
      if constexpr (ES == 4) {
        x = *reinterpret_cast<float*>(el);
        *reinterpret_cast<float*>(el) = -INFINITY;
      } else {
        x = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<unsigned short*>(el)) << 16);
        *reinterpret_cast<unsigned short*>(el) = static_cast<unsigned short>(0xff80u);
      }
      xp = ex2(fmaf(x, c, -d.lp2));
    }
    sm_xp[e] = xp;
  }
  __syncthreads();
  // Per-vector and per-chunk sums of w (the masked copy): vectors tid,
  // tid + 256, ... (the vector sums stay for the pick)
  {
    float sw[kTwMaxChunks];
#pragma unroll
    for (int ci = 0; ci < kTwMaxChunks; ++ci) {
      sw[ci] = 0.f;
      if (ci < nloc) {
        const int lo = (k0 + ci) * ce, hi = min(a.V, lo + ce);
        const int nvec = (hi - lo + NV - 1) / NV;
        const uint4* cv = reinterpret_cast<const uint4*>(chunks + ci * kK3ChunkBytes);
#pragma unroll
        for (int i = 0; i < kTwVecsPerThread; ++i) {
          const int v = i * kTwThreads + tid;
          float av = 0.f;
          if (v < nvec) {
            float x[NV];
            Elem<ES>::unpack(cv[v], x);
#pragma unroll
            for (int e = 0; e < NV; ++e) av += ex2(fmaf(x[e], c, -d.lp2));
          }
          s_vsum[ci * kTwVecs + v] = av;
          sw[ci] += av;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sw[ci] += __shfl_xor_sync(0xffffffffu, sw[ci], o);
      if (lane == 0 && ci < nloc) s_red[ci][warp] = sw[ci];
    }
  }
  __syncthreads();
  if (tid < nloc * kTwCluster) {   // thread (chunk ci, destination CTA r)
    const int ci = tid / kTwCluster, r = tid - ci * kTwCluster;
    const int lo = (k0 + ci) * ce, hi = lo + ce;
    float cw = 0.f, xp = 0.f;
#pragma unroll
    for (int q = 0; q < kTwWarps; ++q) cw += s_red[ci][q];
    for (int e = 0; e < nex; ++e) {
      const int t = s_excl[e];
      if (t >= lo && t < hi) xp += sm_xp[e];
    }
    float2 v = make_float2(cw, cw + xp);
    if (s_err) v = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    st_cluster(map_rank(smem_u32(&s_csum[k0 + ci]), r), v);
  }
  cluster_sync();   // barrier 2: every CTA holds every chunk's sums

  // ---- 4. the chunk holding u * S (every CTA finds the same one). Lane l
  // holds chunks l and l + 32; inclusive scans of the chunk sums give the
  // totals and the crossing together.
  if (warp == 0) {
    const float2 c0 = lane < w.P ? s_csum[lane] : make_float2(0.f, 0.f);
    const float2 c1 = lane + 32 < w.P ? s_csum[lane + 32] : make_float2(0.f, 0.f);
    float iw0 = c0.x, ip0 = c0.y, iw1 = c1.x, ip1 = c1.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float a0 = __shfl_up_sync(0xffffffffu, iw0, o), b0 = __shfl_up_sync(0xffffffffu, ip0, o);
      const float a1 = __shfl_up_sync(0xffffffffu, iw1, o), b1 = __shfl_up_sync(0xffffffffu, ip1, o);
      if (lane >= o) {
        iw0 += a0;
        ip0 += b0;
        iw1 += a1;
        ip1 += b1;
      }
    }
    iw1 += __shfl_sync(0xffffffffu, iw0, 31);
    ip1 += __shfl_sync(0xffffffffu, ip0, 31);
    const float sw = __shfl_sync(0xffffffffu, iw1, 31), sp = __shfl_sync(0xffffffffu, ip1, 31);
    const int usep = !(sw > 0.f);   // no mass left after the removals: draw from p
    const float S = usep ? sp : sw;
    const float thr = d.u * S;
    const float a0 = usep ? c0.y : c0.x, a1 = usep ? c1.y : c1.x;
    const float i0 = usep ? ip0 : iw0, i1 = usep ? ip1 : iw1;
    const float x0 = i0 - a0, x1 = i1 - a1;   // exclusive prefixes
    const unsigned h0 = __ballot_sync(0xffffffffu, lane < w.P && i0 > thr);
    const unsigned h1 = __ballot_sync(0xffffffffu, lane + 32 < w.P && i1 > thr);
    const unsigned g0 = __ballot_sync(0xffffffffu, lane < w.P && a0 > 0.f);
    const unsigned g1 = __ballot_sync(0xffffffffu, lane + 32 < w.P && a1 > 0.f);
    // the first chunk whose inclusive prefix passes u * S; else (rounding)
    // the last chunk with weight; else the last chunk
    int cstar = w.P - 1, half = -1, l = 0;
    if (h0 | h1) {
      half = h0 ? 0 : 1;
      l = __ffs(h0 ? h0 : h1) - 1;
    } else if (g0 | g1) {
      half = g1 ? 1 : 0;
      l = 31 - __clz(g1 ? g1 : g0);
    }
    const float pre0 = __shfl_sync(0xffffffffu, x0, l), pre1 = __shfl_sync(0xffffffffu, x1, l);
    float pre = 0.f;
    if (half >= 0) {
      cstar = half * 32 + l;
      pre = half ? pre1 : pre0;
    }
    if (lane == 0) {
      s_chunk = cstar;
      s_usep = usep | (S == S ? 0 : 2);   // bit 1: a chunk sum was NaN (a wait gave up)
      s_thr = thr - pre;
      s_S = S;
    }
  }
  // a copy that a given-up wait left in flight lands before the CTA exits
  if (s_err && tid == 0) (void)mbar_wait_bounded(smem_u32(&s_bar), 0);
  __syncthreads();
  const int cstar = s_chunk;
  if (cstar < k0 || cstar >= k0 + nloc) return;   // another CTA holds the drawn chunk

  // ---- 5. the owner: the element of the chunk where u * S falls
  const int ci = cstar - k0;
  const int lo = cstar * ce, hi = min(a.V, lo + ce);
  const int nvec = (hi - lo + NV - 1) / NV;
  const int usep = s_usep & 1;
  const float thr = s_thr;
  uint8_t* cs = chunks + ci * kK3ChunkBytes;
  const uint4* cv = reinterpret_cast<const uint4*>(cs);
  float* vs = s_vsum + ci * kTwVecs;
  auto weights = [&](int v, float (&wv)[NV]) {   // the weights of vector v, in element order
    float x[NV];
    Elem<ES>::unpack(cv[v], x);
#pragma unroll
    for (int e = 0; e < NV; ++e) wv[e] = ex2(fmaf(x[e], c, -d.lp2));
  };
  if (usep && nex) {   // drawing from p: the rejected tokens count again
    for (int e = tid; e < nex; e += kTwThreads) {
      const int t = s_excl[e];
      if (t >= lo && t < hi) {
        if constexpr (ES == 4) reinterpret_cast<float*>(cs)[t - lo] = Elem<4>::load(trow, t);
        else reinterpret_cast<unsigned short*>(cs)[t - lo] = __ldg(reinterpret_cast<const unsigned short*>(trow) + t);
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTwVecsPerThread; ++i) {
      const int v = i * kTwThreads + tid;
      float av = 0.f;
      if (v < nvec) {
        float wv[NV];
        weights(v, wv);
#pragma unroll
        for (int e = 0; e < NV; ++e) av += wv[e];
      }
      vs[v] = av;
    }
    __syncthreads();
  }
  // Thread t holds vectors 4t .. 4t + 3 (index order). Block exclusive scan
  // of the thread sums; then each thread's running prefix over its four
  // vectors (the same additions the crossing test below repeats).
  const float4 q4 = reinterpret_cast<const float4*>(vs)[tid];
  const float av[kTwVecsPerThread] = {q4.x, q4.y, q4.z, q4.w};
  float tsum = 0.f;
#pragma unroll
  for (int k = 0; k < kTwVecsPerThread; ++k) tsum += av[k];
  float incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  float ex = 0.f;
  for (int q = 0; q < warp; ++q) ex += s_wsum[q];
  ex += incl - tsum;
  float run = ex;
#pragma unroll
  for (int k = 0; k < kTwVecsPerThread; ++k) run += av[k];
  const unsigned hit = __ballot_sync(0xffffffffu, run > thr && tsum > 0.f);
  const unsigned pos = __ballot_sync(0xffffffffu, tsum > 0.f);
  if (lane == 0) {
    s_cand[warp] = hit ? warp * 32 + __ffs(hit) - 1 : INT_MAX;
    s_wlast[warp] = pos ? warp * 32 + 31 - __clz(pos) : -1;
  }
  __syncthreads();
  int pick = INT_MAX, lastt = -1;
#pragma unroll
  for (int q = 0; q < kTwWarps; ++q) {
    pick = min(pick, s_cand[q]);
    lastt = max(lastt, s_wlast[q]);
  }
  // The drawn element: the first whose inclusive prefix passes u * S; with
  // no crossing (rounding), the last element with weight; else the chunk's
  // last element.
  int j_out = -1;
  if (pick != INT_MAX ? tid == pick : tid == lastt) {
    const bool cross = pick != INT_MAX;
    float r = ex;
    int ksel = -1;
#pragma unroll
    for (int k = 0; k < kTwVecsPerThread; ++k) {
      if (cross) {
        if (ksel < 0) {
          if (r + av[k] > thr && av[k] > 0.f) ksel = k;
          else r += av[k];
        }
      } else if (av[k] > 0.f) {
        ksel = k;
      }
    }
    if (ksel >= 0) {   // always, by construction; guarded for safety
      const int v = 4 * tid + ksel;
      float wv[NV];
      weights(v, wv);
      float part = 0.f;
      int e_sel = -1, e_last = -1;
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        part += wv[e];
        if (wv[e] > 0.f) e_last = e;
        if (cross && e_sel < 0 && r + part > thr && wv[e] > 0.f) e_sel = e;
      }
      j_out = lo + v * NV + (e_sel >= 0 ? e_sel : e_last);
    }
  } else if (pick == INT_MAX && lastt < 0 && ((hi - 1 - lo) / NV) / kTwVecsPerThread == tid) {
    j_out = hi - 1;
  }
  if (j_out >= 0) {
    float x_out;
    if constexpr (ES == 4) x_out = reinterpret_cast<const float*>(cs)[j_out - lo];
    else x_out = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short*>(cs)[j_out - lo]) << 16);
    if (x_out == -INFINITY) x_out = Elem<ES>::load(trow, j_out);   // a masked element (no weight anywhere)
    const float p = ex2(fmaf(x_out, c, -d.lp2));
    const int64_t o = static_cast<int64_t>(b) * W + d.pos;
    a.out_tokens[o] = j_out;
    if (a.out_logprob) a.out_logprob[o] = (x_out * c - d.lp2) * kLn2;
    if (a.out_mu) a.out_mu[o] = d.type == kDrawMaskedP ? d.scale * p / s_S : p;
    if (a.out_status) a.out_status[b] = d.status | ((s_usep & 2) ? kStatusWaitErr : 0);
  }
  if (a.fin.out_len) {   // this kernel ends the call
    __syncthreads();
    finish_request(a.fin, fpre, s_stop, b, d.pos, W, a.out_tokens, a.out_logprob, a.out_mu, a.out_nodes,
                   a.out_status, s_fin);
  }
}

}  // namespace sv
