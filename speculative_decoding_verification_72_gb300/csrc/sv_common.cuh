// Device helpers shared by the verification kernels: inline PTX for mbarriers,
// 1-D bulk (TMA) copies, the SFU exp2, programmatic dependent launch, and the
// per-(row, segment) partial record of the row-streaming pass.
#pragma once

#include <cstdint>
#include <climits>
#include <cfloat>
#include <cuda_runtime.h>

// Status bits and return codes are the C ABI's (include/spec_verify.h), so
// kernels and header cannot drift apart.
#include "spec_verify.h"

namespace sv {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

// Partial statistics of one segment of one logit row. With c = log2(e) / T:
//   m   = max x_j over the segment (raw logits; -inf if no element > -inf)
//   s   = sum_j 2^((x_j - m) c)           (0 when m = -inf)
//   idx = lowest row-relative index with x_j == m (INT_MAX if none)
//   err = nonzero if a bounded wait in the producing CTA gave up
struct __align__(16) Partial {
  float m;
  float s;
  int32_t idx;
  int32_t err;
};

// Output position the residual / bonus draw of one request fills, and how.
enum DrawType : int32_t {
  kDrawNone = 0,
  kDrawP = 1,        // w = p
  kDrawMaskedP = 2,  // w = p with the listed tokens removed
  kDrawResid = 3,    // w = relu(p - q)
};

struct __align__(16) DrawDesc {
  int32_t type;    // DrawType
  int32_t t_row;   // global target row
  int32_t d_row;   // global draft row (kDrawResid)
  int32_t pos;     // output column
  float u;         // caller's uniform for this draw
  float lp2;       // log2-domain lse of the target row: m c + log2(s)
  float lq2;       // same for the draft row
  float scale;     // probability of reaching this draw (kDrawMaskedP)
  int32_t n_excl;  // tokens removed (kDrawMaskedP)
  int32_t pad0, pad1, pad2;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// SFU base-2 exponential (PTX ex2.approx.ftz.f32): relative error ~2^-22,
// -inf -> +0, results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// SFU base-2 logarithm (PTX lg2.approx.ftz.f32): absolute error ~2^-22 in
// the result; +0 -> -inf.
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// --------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up and returns false after kWaitNs
// of polling (or kWaitIters polls); it never spins forever. The time between
// two polls is counted at most kWaitGapNs, so a context that is switched out
// while it waits (time-slicing with another process, compute preemption) does
// not give up early because the global timer ran on meanwhile.
constexpr uint64_t kWaitNs = 20ull * 1000ull * 1000ull;  // 20 ms of polling
constexpr uint64_t kWaitGapNs = 1000ull * 1000ull;      // 1 ms
constexpr uint32_t kWaitIters = 1u << 22;

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t prev = global_timer_ns(), spent = 0;
  for (uint32_t it = 1; it < kWaitIters; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t now = global_timer_ns();
    const uint64_t gap = now - prev;
    spent += gap < kWaitGapNs ? gap : kWaitGapNs;
    prev = now;
    if (spent > kWaitNs) return false;
  }
  return false;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (a hint: no data reaches the
// program). src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Store of one Partial that asks L2 to keep the line (evict_last): the
// decide kernels read the partials after the row pass, which meanwhile
// streams far more than L2 holds, and partials written early in it would
// otherwise have left L2 by then.
__device__ __forceinline__ void store_partial_keep(Partial* dst, const Partial& v) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "r"(__float_as_uint(v.m)),
               "r"(__float_as_uint(v.s)), "r"(static_cast<uint32_t>(v.idx)), "r"(static_cast<uint32_t>(v.err)), "l"(pol)
               : "memory");
}

// Warp-wide maximum of a float in one instruction (redux.sync, sm_100 and
// later). NaN inputs are ignored, as with fmaxf.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Warp-wide minimum of a non-negative int in one instruction.
__device__ __forceinline__ int warp_min_nonneg(int v) {
  uint32_t r;
  asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(static_cast<uint32_t>(v)));
  return static_cast<int>(r);
}

// Barrier over a subset of the CTA's warps (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------ programmatic dependent launch

// Wait until the preceding kernel in the stream has completed and its writes
// are visible (no-op when launched without the programmatic attribute).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the dependent kernel to begin launching.
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ element types

template <int ES>
struct Elem;

template <>
struct Elem<4> {  // fp32
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float load(const uint8_t* row, int j) {
    return __ldg(reinterpret_cast<const float*>(row) + j);
  }
  __device__ __forceinline__ static void unpack(const uint4& w, float* f) {
    f[0] = __uint_as_float(w.x);
    f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z);
    f[3] = __uint_as_float(w.w);
  }
};

template <>
struct Elem<2> {  // bf16: the value is the high half of an fp32
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float load(const uint8_t* row, int j) {
    const unsigned short v = __ldg(reinterpret_cast<const unsigned short*>(row) + j);
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  __device__ __forceinline__ static void unpack(const uint4& w, float* f) {
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
    f[4] = __uint_as_float(w.z << 16);
    f[5] = __uint_as_float(w.z & 0xffff0000u);
    f[6] = __uint_as_float(w.w << 16);
    f[7] = __uint_as_float(w.w & 0xffff0000u);
  }
};

// --------------------------------------------------- online max / sum-exp

// Combine partial (m2, s2, i2) into (m, s, i): max, rescaled sum, lowest
// index on equal maxima. Symmetric, so any fixed reduction order is
// deterministic.
__device__ __forceinline__ void merge_stats(float& m, float& s, int& i, float m2, float s2, int i2,
                                            float c) {
  if (m2 > m) {
    s = (m == -INFINITY ? 0.f : s * ex2((m - m2) * c)) + s2;
    m = m2;
    i = i2;
  } else if (m2 == m) {
    s += s2;
    i = min(i, i2);
  } else if (m2 != -INFINITY) {
    s += s2 * ex2((m2 - m) * c);
  }
}

}  // namespace sv
