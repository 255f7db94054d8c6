// Early-exit row statistics for greedy chains (mini-sglang PR #134,
// verify.py: the accepted prefix ends at the first draft that differs from
// its row's argmax, and rows after that row never reach the outputs).
//
// The same TMA ring, stage fold and piece merge as row_stats_kernel, with a
// different schedule: each CTA takes whole rows, cyclically, in
// position-major order (position i of every request before position i + 1),
// so the low positions of all requests are read first. The CTA that finishes
// row i of request b compares its argmax with draft i and, on a mismatch,
// raises state[b] to 0x7fffffff - i (an atomic max, so the smallest known
// mismatching position wins); then it counts the row in done[b]. Before
// streaming row i of request b the producer reads state[b] and skips the row
// when a mismatch is known at a smaller position. A row of a later wave (the
// rows k in [w G, (w + 1) G) form wave w) first waits, boundedly, until
// done[b] covers the request's rows in the earlier waves or a mismatch before
// it is known: the rows of a wave land at about the same time, so without the
// wait a CTA would read its next row before the earlier wave's mismatches are
// published. Every skipped row lies after a known mismatch, so the wait ends;
// if it hits its limit the row is read. No row at or before a request's first mismatch is ever
// skipped, so the decide kernel sees exactly the statistics it needs; rows
// after it may be skipped and their partial slots keep stale values, which
// the decide kernel never uses. A CTA whose bounded waits gave up marks its
// byte count (top bit), and the decide kernel then reports TIMEOUT.
//
// The producer decides which rows are read, so each ring slot carries the
// row and stage it holds (written before the slot's full barrier is armed,
// which publishes it to the consumers); the consumers follow those stage
// descriptors instead of recomputing the schedule, and an end marker closes
// the stream. One Partial per row, at slot `row`. Each CTA writes the bytes
// it requested to cta_bytes[g].
#pragma once

#include "decide.cuh"
#include "row_stats.cuh"

namespace sv {

struct EarlyArgs {
  RowStatsArgs rs;            // target rows only; rs.partials: slot = row
  int32_t B, R;               // requests, rows per request (K + 1)
  const int32_t* drafts;      // [B, K]
  int32_t* state;             // [B]: 0, or 0x7fffffff - (smallest known mismatching position)
  int32_t* done;              // [B]: rows of the request finished in this call
  unsigned long long* cta_bytes;  // [G]
};

__device__ __forceinline__ int ld_relaxed(const int32_t* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Polling limit of the wave gate (a performance wait: when it runs out the
// row is simply read).
constexpr uint64_t kWaveGateNs = 200ull * 1000ull;   // 200 us

template <int ES>
__global__ void __maxnreg__(kK1MaxRegs) row_stats_early_kernel(const EarlyArgs e) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[kK1Stages];
  __shared__ __align__(8) uint64_t empty_bar[kK1Stages];
  __shared__ Partial red[kK1RedBufs][kK1Consumers];
  __shared__ int red_cnt[kK1RedBufs];
  __shared__ int meta_row[kK1Stages];   // row in the slot, -1 = end of stream
  __shared__ int meta_sg[kK1Stages];    // stage of that row
  __shared__ int meta_nst[kK1Stages];   // stages of that row (0: scalar elements only)

  const RowStatsArgs& a = e.rs;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x;
  const int rows = e.B * e.R;

  if (tid < kK1RedBufs) red_cnt[tid] = 0;   // shared-memory setup overlaps the previous kernel
  if (tid == 0) {
    for (int i = 0; i < kK1Stages; ++i) {
      mbar_init(smem_u32(&full_bar[i]), 1);
      mbar_init(smem_u32(&empty_bar[i]), kK1Consumers);
    }
    fence_barrier_init();
  }
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The warp checks the CTA's next 32 rows against the state words at once
    // (one load per lane); lane 0 streams the first row still needed, and
    // the rows after it get a fresh check. Skipped rows cost a round trip
    // per 32, not one each.
    int st = 0, slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    unsigned long long bytes = 0;
    // Take a free slot (its previous use released) and describe it.
    auto claim = [&](int row, int sg, int nst) -> bool {
      if (st >= kK1Stages && !mbar_wait_bounded(smem_u32(&empty_bar[slot]), phase ^ 1)) return false;
      meta_row[slot] = row;
      meta_sg[slot] = sg;
      meta_nst[slot] = nst;
      return true;
    };
    auto advance = [&]() {
      ++st;
      if (++slot == kK1Stages) {
        slot = 0;
        phase ^= 1;
      }
    };
    // The CTA's rows k = g + j G belong to requests (g + j G) mod B, which
    // repeat with period B / gcd(B, G); positions only grow along the
    // sequence and a request's known mismatch position only falls, so once
    // a checked batch covering a whole period is all skipped, every later
    // row is too.
    int gcd_bg = e.B, rem = a.G % e.B;
    while (rem != 0) {
      const int t = gcd_bg % rem;
      gcd_bg = rem;
      rem = t;
    }
    const bool batch_spans_period = e.B / gcd_bg <= 32;
    int k0 = g;
    while (k0 < rows && ok) {
      const int64_t kl = static_cast<int64_t>(k0) + static_cast<int64_t>(lane) * a.G;
      bool need = false;
      if (kl < rows) {
        const int i = static_cast<int>(kl) / e.B;
        const int sb = ld_relaxed(e.state + (static_cast<int>(kl) - i * e.B));
        need = !(sb != 0 && 0x7fffffff - sb < i);   // no mismatch known before position i
      }
      const unsigned m = __ballot_sync(0xffffffffu, need);
      if (m == 0) {
        if (batch_spans_period && static_cast<long long>(k0) + 31ll * a.G < rows) break;
        const long long nx = static_cast<long long>(k0) + 32ll * a.G;
        k0 = nx < rows ? static_cast<int>(nx) : rows;
        continue;
      }
      const int k = k0 + (__ffs(m) - 1) * a.G;
      k0 = k < rows - a.G ? k + a.G : rows;
      if (lane == 0) {
        const int i = k / e.B;
        const int b = k - i * e.B;
        const int row = b * e.R + i;
        // Wave gate: request b has ceil((wave start - b) / B) rows in the
        // earlier waves; wait for them to finish, or for a mismatch before i.
        const long long ws0 = static_cast<long long>(k / a.G) * a.G;
        const int need_done = ws0 > b ? static_cast<int>((ws0 - b + e.B - 1) / e.B) : 0;
        bool skip = false;
        if (need_done > 0) {
          const uint64_t t0 = global_timer_ns();
          for (int it = 0; it < (1 << 20); ++it) {
            const int sb = ld_relaxed(e.state + b);
            if (sb != 0 && 0x7fffffff - sb < i) {
              skip = true;
              break;
            }
            if (ld_acquire(e.done + b) >= need_done || global_timer_ns() - t0 > kWaveGateNs) break;
            __nanosleep(200);
          }
          if (!skip) {   // a mismatch published just before the last count
            const int sb = ld_relaxed(e.state + b);
            skip = sb != 0 && 0x7fffffff - sb < i;
          }
        }
        if (!skip) {
          const Piece p = make_piece<ES>(a, row, 0, static_cast<int64_t>(row + 1) * a.V);
          bytes += static_cast<unsigned long long>(p.cp_hi - p.cp_lo) +
                   static_cast<unsigned long long>((p.head_end - p.j0) + (p.j1 - p.tail_begin)) * ES;
          if (p.nst == 0) {   // scalar elements only: a descriptor with no copy
            if ((ok = claim(row, 0, 0))) {
              mbar_arrive(smem_u32(&full_bar[slot]));
              advance();
            }
          }
          for (int s = 0; s < p.nst && ok; ++s) {
            if (!(ok = claim(row, s, p.nst))) break;
            const uint32_t off = static_cast<uint32_t>(s) * kK1StageBytes;
            const uint32_t nb = min(static_cast<uint32_t>(kK1StageBytes), static_cast<uint32_t>(p.cp_hi - p.cp_lo) - off);
            const uint32_t fb = smem_u32(&full_bar[slot]);
            mbar_arrive_expect_tx(fb, nb);
            bulk_g2s(smem_u32(ring + slot * kK1StageBytes), reinterpret_cast<const void*>(p.cp_lo + off), nb, fb);
            advance();
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      if (ok) ok = claim(-1, 0, 0);   // end of stream
      if (ok) {
        mbar_arrive(smem_u32(&full_bar[slot]));
        advance();
      }
      for (int k = max(0, st - kK1Stages); k < st; ++k)
        ok = mbar_wait_bounded(smem_u32(&full_bar[k % kK1Stages]), (k / kK1Stages) & 1) && ok;
      // a wait that gave up leaves rows unread: the top bit tells the decide kernel
      e.cta_bytes[g] = ok ? bytes : (bytes | kEarlyAbortBit);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  uint4* const stash = reinterpret_cast<uint4*>(ring + kK1RingBytes);
  const int ct = tid - 32;
  const int cw = warp - 1;
  const float c = a.c;
  const int K = e.R - 1;
  int slot = 0, npiece = 0;
  uint32_t phase = 0;
  bool ok = true;
  float ref = 0.f;
  float m = -INFINITY, mc = 0.f, s = 0.f;
  GroupCand cand;
  Piece p;
  int jbase = 0;
  while (true) {
    if (!mbar_wait_bounded(smem_u32(&full_bar[slot]), phase)) {
      ok = false;   // the producer stops too; nothing more is written
      break;
    }
    const int mrow = meta_row[slot], msg = meta_sg[slot], mnst = meta_nst[slot];
    if (mrow < 0) break;
    if (msg == 0) {   // first stage (or only descriptor) of a row
      p = make_piece<ES>(a, mrow, 0, static_cast<int64_t>(mrow + 1) * a.V);
      m = -INFINITY;
      mc = ref;
      s = 0.f;
      cand.stage = -1;
      cand.vec = 0;
      cand.j = INT_MAX;
      cand.jbase = 0;
      jbase = p.j0 - static_cast<int>((p.lo - p.cp_lo) / ES);
      for (int j = p.j0 + ct; j < p.head_end; j += kK1ConsumerThreads)
        fold_scalar(Elem<ES>::load(p.rowp, j), j, c, m, mc, s, cand);
    }
    if (mnst > 0) {
      uint4* sv4 = reinterpret_cast<uint4*>(ring + slot * kK1StageBytes);
      const int last = mnst - 1;
      const bool first_edge = p.cp_lo < p.lo;
      const bool last_hull = p.cp_hi > p.hi;
      const int last_nvec = static_cast<int>((p.cp_hi - p.cp_lo - static_cast<uintptr_t>(last) * kK1StageBytes) / 16u);
      const bool last_edge = last_hull || last_nvec != kStageFullVecs;
      const int nh = msg == last ? stage_halves(warp - 1, last_nvec) : kStageHalves;
      if ((msg == 0 && first_edge) || (msg == last && last_edge)) {
        const int nvec = msg == last ? last_nvec : kStageFullVecs;
        mask_stage<ES>(sv4, ct, nvec, jbase, p.j0, p.j1, (msg == 0 && first_edge) ? 0 : -1,
                       (msg == last && last_hull) ? nvec - 1 : -1, nh);
      }
      fold_stage_n<ES>(sv4, stash, ct, jbase, msg, c, m, mc, s, cand, nh);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
    jbase += kK1StageBytes / ES;
    if (++slot == kK1Stages) {
      slot = 0;
      phase ^= 1;
    }
    if (mnst > 0 && msg != mnst - 1) continue;

    // ---- end of row mrow: tail elements, then the warp and CTA merge
    for (int j = p.tail_begin + ct; j < p.j1; j += kK1ConsumerThreads)
      fold_scalar(Elem<ES>::load(p.rowp, j), j, c, m, mc, s, cand);
    if (m > -INFINITY) ref = mc;
    const float wm = warp_max(m);
    const int widx = warp_min_nonneg((m == wm) ? resolve_cand<ES>(cand, stash, ct, m, p.j0, p.j1) : INT_MAX);
    float ws = (m == -INFINITY) ? 0.f : s * ex2((m - wm) * c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    const int buf = npiece & (kK1RedBufs - 1);
    ++npiece;
    int merger = 0;
    if (lane == 0) {
      Partial mine;
      mine.m = wm;
      mine.s = ws;
      mine.idx = widx;
      mine.err = ok ? 0 : 1;
      red[buf][cw] = mine;
      __threadfence_block();
      merger = atomicAdd(&red_cnt[buf], 1) == kK1Consumers - 1;
    }
    if (__shfl_sync(0xffffffffu, merger, 0)) {
      __threadfence_block();
      float rm = -INFINITY, rs = 0.f;
      int ri = INT_MAX, re = 0;
      if (lane < kK1Consumers) {
        const Partial v = red[buf][lane];
        rm = v.m;
        rs = v.s;
        ri = v.idx;
        re = v.err;
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, rm, o);
        const float os = __shfl_xor_sync(0xffffffffu, rs, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ri, o);
        re |= __shfl_xor_sync(0xffffffffu, re, o);
        merge_stats(rm, rs, ri, om, os, oi, c);
      }
      if (lane == 0) {
        atomicExch(&red_cnt[buf], 0);
        if (rm == -INFINITY) ri = 0;   // every element -inf: the lowest index attains the max
        Partial out;
        out.m = rm;
        out.s = rs;
        out.idx = ri;
        out.err = re;
        a.partials[mrow] = out;
        // publish a mismatch at this row's position
        const int b = mrow / e.R;
        const int i = mrow - b * e.R;
        if (i < K) {
          const int d = e.drafts[static_cast<int64_t>(b) * K + i];
          if (d < 0 || d >= a.V || d != ri) atomicMax(e.state + b, 0x7fffffff - i);
        }
        __threadfence();   // the partial and the mismatch before the count
        atomicAdd(e.done + b, 1);
      }
    }
  }
}

}  // namespace sv
