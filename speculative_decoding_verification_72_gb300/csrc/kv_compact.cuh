// Accepted-path KV compaction, the step after tree verification (nanospec
// README: paged KV cache, EAGLE-3 tree speculation; mini-sglang PR #134,
// draft.py: the cache keeps the accepted prefix, the rest is truncated).
//
// The verify pass wrote node n's key/value row at logical position
// seq_base[b] + n; logical position p lives at slot p % P of page
// page_table[b, p / P] of a cache laid out [pages, P, row] (rows
// token_stride bytes apart). The accepted path path_nodes[b, 0..n] (node 0
// the root) moves so that its j-th node lands at position seq_base[b] + j, and
// the committed length becomes seq_base[b] + n + 1.
//
// Grid = B x chunks; CTA (b, c) moves bytes [c * 4 KB, (c + 1) * 4 KB) of
// every path row of request b, 16 bytes per thread per row. Path nodes
// strictly increase (a parent precedes its child), so a destination j never
// holds a later step's source (path_nodes[j'] >= j' > j): steps are taken in
// increasing j, kKvStepBatch at a time, each batch's loads issued before its
// stores, one round trip per batch. Every CTA of a request validates the
// whole path first (node ids, page ids), so a bad request is left untouched
// by all of them.
#pragma once

#include "sv_common.cuh"

namespace sv {

constexpr int kKvThreads = 256;
constexpr int kKvChunkBytes = kKvThreads * 16;
constexpr int kKvStepBatch = 8;
constexpr int kStatusBadPage = SV_STATUS_BAD_PAGE;

struct KvCompactArgs {
  uint8_t* kv;
  int64_t token_stride;        // bytes between consecutive slots of a page
  int64_t page_bytes;          // page_size * token_stride
  int32_t row_bytes;           // bytes of one token row (multiple of 16)
  const int32_t* page_table;   // [B, max_pages]
  int32_t max_pages, page_size;
  const int32_t* seq_base;     // [B]
  const int32_t* path_nodes;   // [B, path_cols]
  int32_t path_cols;
  const int32_t* num_accepted; // [B]
  int32_t max_nodes;           // node ids must lie in [0, max_nodes)
  int32_t chunks;              // ceil(row_bytes / kKvChunkBytes)
  int32_t* out_len;            // [B]
  int32_t* out_status;         // [B] or nullptr
};

// Byte offset of logical position p of request b, or -1 if its page is invalid.
__device__ __forceinline__ int64_t kv_offset(const KvCompactArgs& a, int b, int64_t p) {
  if (p < 0) return -1;
  const int64_t lp = p / a.page_size;
  if (lp >= a.max_pages) return -1;
  const int page = a.page_table[static_cast<int64_t>(b) * a.max_pages + lp];
  if (page < 0) return -1;
  return static_cast<int64_t>(page) * a.page_bytes + (p - lp * a.page_size) * a.token_stride;
}

__global__ void __launch_bounds__(kKvThreads) kv_compact_kernel(const KvCompactArgs a) {
  __shared__ int64_t s_src[kKvStepBatch], s_dst[kKvStepBatch];
  grid_dep_wait();   // the path and n come from the verify call before this kernel
  grid_dep_launch();
  const int b = blockIdx.x / a.chunks;
  const int ch = blockIdx.x - b * a.chunks;
  const int tid = threadIdx.x;
  const int32_t* nodes = a.path_nodes + static_cast<int64_t>(b) * a.path_cols;
  // The count and the thread's first path entry are loaded together (the
  // entry is inside the row whatever the count is).
  const int v_first = tid < a.path_cols ? nodes[tid] : 0;
  const int n = a.num_accepted[b];
  const int64_t base = a.seq_base[b];
  // validate the whole path (every CTA of the request reaches the same answer)
  bool ok = n >= 0 && n < a.path_cols;
  if (ok) {
    for (int j = tid; j <= n; j += kKvThreads) {
      const int v = j == tid ? v_first : nodes[j];
      ok = ok && v >= 0 && v < a.max_nodes && kv_offset(a, b, base + v) >= 0 && kv_offset(a, b, base + j) >= 0;
    }
  }
  ok = __syncthreads_and(ok);
  if (ch == 0 && tid == 0) {
    a.out_len[b] = ok ? static_cast<int32_t>(base + n + 1) : static_cast<int32_t>(base);
    if (a.out_status) a.out_status[b] = ok ? 0 : kStatusBadPage;
  }
  if (!ok) return;
  const int64_t off = static_cast<int64_t>(ch) * kKvChunkBytes + static_cast<int64_t>(tid) * 16;
  const bool mine = off < a.row_bytes;
  for (int j0 = 0; j0 <= n; j0 += kKvStepBatch) {
    __syncthreads();   // the previous batch's addresses are no longer read
    if (tid < kKvStepBatch) {
      const int j = j0 + tid;
      int64_t src = -1, dst = -1;
      if (j <= n) {
        const int v = nodes[j];
        if (v != j) {   // a node already in place does not move
          src = kv_offset(a, b, base + v);
          dst = kv_offset(a, b, base + j);
        }
      }
      s_src[tid] = src;
      s_dst[tid] = dst;
    }
    __syncthreads();
    if (!mine) continue;
    uint4 buf[kKvStepBatch];
#pragma unroll
    for (int t = 0; t < kKvStepBatch; ++t)
      if (s_src[t] >= 0) buf[t] = *reinterpret_cast<const uint4*>(a.kv + s_src[t] + off);
#pragma unroll
    for (int t = 0; t < kKvStepBatch; ++t)
      if (s_src[t] >= 0) *reinterpret_cast<uint4*>(a.kv + s_dst[t] + off) = buf[t];
  }
}

}  // namespace sv
