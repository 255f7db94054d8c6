// Host side of the libspecverify C ABI (include/spec_verify.h): argument
// validation, the workspace plan shared by the *_workspace_size functions and
// the launchers, and the kernel launches.
//
// One call is K1 (row statistics) [-> top-k bound] -> K2 (decide) [-> K3
// (draw) [-> mu pass]] on the caller's stream; the bracketed kernels run only
// for the rules that need them (rules.cuh). Every kernel is launched with
// programmatic stream serialization, so its launch overlaps the tail of the
// kernel before it. K1 waits (griddepcontrol.wait) before reading anything,
// so the logits may come from the kernel just before the call; the others
// read only the call's own inputs before their wait and earlier kernels'
// results after it (the top-k kernel waits first, so a wait on it also
// covers K1).

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "spec_verify.h"
#include "decide.cuh"
#include "draw.cuh"
#include "row_stats.cuh"
#include "row_stats_early.cuh"
#include "rules.cuh"
#include "tree_build.cuh"
#include "tree_draw.cuh"
#include "kv_compact.cuh"
#include "selftest.cuh"

namespace {

using namespace sv;

constexpr size_t kAlign = 256;
static_assert(SV_MAX_STOP_IDS == kMaxStopIds, "stop ids staged in shared memory");

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elem_size(int32_t dtype) {
  if (dtype == SV_F32) return 4;
  if (dtype == SV_BF16) return 2;
  return 0;
}

struct Plan {
  int64_t rows_total = 0;
  int64_t T = 0;            // rows_total * V, K1's flattened element count
  int32_t P = 0;            // K3 chunks per row
  int32_t chunk_elems = 0;
  int32_t excl_stride = 0;
  size_t off_part = 0, off_draw = 0, off_excl = 0, off_k3part = 0;
  size_t off_thr = 0, off_mupart = 0, off_mucnt = 0;
  size_t total = 0;
};

// Workspace layout; independent of the device (K1's partial array is sized
// for the largest grid K1 may use, kK1MaxCtas). Stochastic calls also hold a
// rank bound per target row and, with draft logits (mu_rows = B * K > 0), the
// mu pass's chunk sums and tickets, whatever rule the call uses.
bool make_plan(int64_t rows_t, int64_t rows_d, int64_t B, int64_t V, int es, bool draw,
               int64_t excl_stride, int64_t mu_rows, Plan* pl) {
  if (V < 1 || es == 0 || B < 0 || rows_t < 0 || rows_d < 0) return false;
  pl->chunk_elems = kK3ChunkBytes / es;
  pl->P = static_cast<int32_t>((V + pl->chunk_elems - 1) / pl->chunk_elems);
  pl->rows_total = rows_t + rows_d;
  if (pl->rows_total > INT32_MAX / 2) return false;
  pl->T = pl->rows_total * V;
  if (draw && B * pl->P >= INT32_MAX) return false;
  if (mu_rows * pl->P >= INT32_MAX) return false;
  pl->excl_stride = static_cast<int32_t>(excl_stride < 1 ? 1 : excl_stride);
  size_t off = 0;
  pl->off_part = off;
  // one partial per (row piece, consumer warp): (rows + G) * kK1Consumers slots
  off += align_up(static_cast<size_t>(pl->rows_total + kK1MaxCtas) * kK1Consumers * sizeof(Partial), kAlign);
  if (draw) {
    pl->off_draw = off;
    off += align_up(static_cast<size_t>(B) * sizeof(DrawDesc), kAlign);
    pl->off_excl = off;
    off += align_up(static_cast<size_t>(B) * pl->excl_stride * sizeof(int32_t), kAlign);
    pl->off_k3part = off;
    off += align_up(static_cast<size_t>(B) * pl->P * sizeof(float2), kAlign);
    pl->off_thr = off;
    off += align_up(static_cast<size_t>(rows_t) * sizeof(float), kAlign);
    if (mu_rows > 0) {
      pl->off_mupart = off;
      off += align_up(static_cast<size_t>(mu_rows) * pl->P * sizeof(float2), kAlign);
      pl->off_mucnt = off;
      off += align_up(static_cast<size_t>(B) * sizeof(uint32_t), kAlign);
    }
  }
  pl->total = off < kAlign ? kAlign : off;
  return true;
}

// Per-device facts looked up once (SM count, kernel attributes set). Reads
// take an atomic fast path; the first lookup on a device runs under a mutex,
// so concurrent first calls from several host threads are safe. Devices past
// kMaxDevices are not cached (looked up on every call).
constexpr int kMaxDevices = 64;
std::mutex g_dev_cache_mu;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<uint32_t> g_attr_done[kMaxDevices];

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// SM count of the current device.
int sm_count() {
  const int dev = current_device();
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached) {
    const int n = g_sm_count[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
  }
  std::lock_guard<std::mutex> lock(g_dev_cache_mu);
  if (cached && g_sm_count[dev].load(std::memory_order_relaxed) > 0) return g_sm_count[dev].load();
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (cached) g_sm_count[dev].store(n, std::memory_order_release);
  return n;
}

// Runs `set` (kernel attribute calls) once per device for the attribute group
// `bit`; a failed attempt is retried on the next call.
enum AttrBit : uint32_t { kAttrK1 = 1, kAttrK1Early = 2, kAttrRowTopk = 4, kAttrDraw = 8, kAttrTreeDraw = 16 };

template <typename F>
cudaError_t once_per_device(uint32_t bit, F&& set) {
  const int dev = current_device();
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && (g_attr_done[dev].load(std::memory_order_acquire) & bit)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_dev_cache_mu);
  if (cached && (g_attr_done[dev].load(std::memory_order_relaxed) & bit)) return cudaSuccess;
  const cudaError_t e = set();
  if (e == cudaSuccess && cached) g_attr_done[dev].fetch_or(bit, std::memory_order_release);
  return e;
}

// Largest dynamic shared memory and the largest shared-memory carveout, so
// two rings fit on one SM.
template <typename Kern>
cudaError_t set_smem_attrs(Kern kernel, int smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

// K1 grid for this device: kK1CtasPerSm per SM, fewer for small problems.
int k1_grid(int64_t T, int es) {
  int64_t g = static_cast<int64_t>(sm_count()) * kK1CtasPerSm;
  const int64_t by_size = (T * es + kK1MinBytesPerCta - 1) / kK1MinBytesPerCta;
  if (by_size < g) g = by_size;
  if (g > kK1MaxCtas) g = kK1MaxCtas;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_temperature(float t) { return std::isfinite(t) && t >= 1e-4f; }

sv_status check_rule(const sv_rule_params& r) {
  if (r.rule != SV_RULE_EXACT && r.rule != SV_RULE_RELAXED && r.rule != SV_RULE_POWER)
    return SV_ERR_INVALID_ARG;
  if (r.rule == SV_RULE_POWER && !(std::isfinite(r.alpha) && r.alpha > 0.f)) return SV_ERR_INVALID_ARG;
  if (r.rule == SV_RULE_RELAXED) {
    if (std::isnan(r.tau)) return SV_ERR_INVALID_ARG;
    if (r.top_k < 0 || r.top_k > SV_MAX_TOP_K) return SV_ERR_INVALID_ARG;
  }
  return SV_OK;
}

RuleArgs rule_args(const sv_rule_params& r) {
  RuleArgs a;
  a.rule = r.rule;
  a.tau = r.tau;
  a.top_k = r.rule == SV_RULE_RELAXED ? r.top_k : 0;
  a.alpha = r.rule == SV_RULE_POWER ? r.alpha : 1.f;
  a.thr = nullptr;
  return a;
}

template <typename Kern, typename Args>
cudaError_t launch(Kern kernel, int grid, int block, size_t smem, cudaStream_t stream, bool pdl,
                   const Args& args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

template <int ES>
cudaError_t launch_row_stats(const RowStatsArgs& a, cudaStream_t stream) {
  const cudaError_t e = once_per_device(kAttrK1 << (ES == 2 ? 0 : 8),
                                        [] { return set_smem_attrs(row_stats_kernel<ES>, kK1SmemBytes); });
  if (e != cudaSuccess) return e;
  return launch(row_stats_kernel<ES>, a.G, kK1Threads, kK1SmemBytes, stream, true, a);
}

template <int ES>
cudaError_t launch_row_stats_early(const EarlyArgs& e, cudaStream_t stream) {
  const cudaError_t err = once_per_device(kAttrK1Early << (ES == 2 ? 0 : 8),
                                          [] { return set_smem_attrs(row_stats_early_kernel<ES>, kK1SmemBytes); });
  if (err != cudaSuccess) return err;
  return launch(row_stats_early_kernel<ES>, e.rs.G, kK1Threads, kK1SmemBytes, stream, true, e);
}

cudaError_t launch_topk(const void* tgt, int64_t stride_b, int32_t rows_per_req, int32_t row_pitch,
                        int32_t V, int32_t k, const int32_t* parents, float* thr, int64_t grid, int es,
                        cudaStream_t st) {
  TopkArgs t;
  t.tgt = static_cast<const uint8_t*>(tgt);
  t.tgt_stride = stride_b;
  t.rows_per_req = rows_per_req;
  t.row_pitch = row_pitch;
  t.V = V;
  t.k = k;
  t.parents = parents;
  t.thr = thr;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  return es == 2 ? launch(topk_threshold_kernel<2>, static_cast<int>(grid), kTkThreads, 0, st, true, t)
                 : launch(topk_threshold_kernel<4>, static_cast<int>(grid), kTkThreads, 0, st, true, t);
}

RowSet row_set(const void* base, int64_t stride_elems, int64_t rows, int64_t V, int es) {
  RowSet r;
  r.base = static_cast<const uint8_t*>(base);
  r.stride_bytes = stride_elems * es;
  r.rows = static_cast<int32_t>(rows);
  r.safe_lo = reinterpret_cast<uintptr_t>(base);
  r.safe_hi = rows > 0 ? r.safe_lo + static_cast<uintptr_t>(((rows - 1) * stride_elems + V) * es) : r.safe_lo;
  return r;
}

RowStatsArgs row_stats_args(const Plan& pl, const void* tgt, int64_t tgt_stride, int64_t rows_t,
                            const void* dft, int64_t dft_stride, int64_t rows_d, int32_t V, int es,
                            float c, void* ws) {
  RowStatsArgs r;
  r.set0 = row_set(tgt, tgt_stride, rows_t, V, es);
  r.set1 = row_set(dft, dft_stride, rows_d, V, es);
  r.V = V;
  r.T = pl.T;
  r.G = k1_grid(pl.T, es);
  r.c = c;
  r.partials = reinterpret_cast<Partial*>(static_cast<uint8_t*>(ws) + pl.off_part);
  return r;
}

DrawArgs draw_args(const Plan& pl, const void* tgt, int64_t tgt_stride, int64_t rows_t, const void* dft,
                   int64_t dft_stride, int64_t rows_d, int32_t B, int32_t V, int es, float c, void* ws,
                   int32_t out_cols, int32_t* out_tokens, float* out_logprob, float* out_mu) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  const RowSet t = row_set(tgt, tgt_stride, rows_t, V, es);
  const RowSet d0 = row_set(dft, dft_stride, rows_d, V, es);
  DrawArgs d;
  std::memset(&d, 0, sizeof(d));
  d.tgt = t.base;
  d.tgt_stride = t.stride_bytes;
  d.tgt_lo = t.safe_lo;
  d.tgt_hi = t.safe_hi;
  d.dft = d0.base;
  d.dft_stride = d0.stride_bytes;
  d.dft_lo = d0.safe_lo;
  d.dft_hi = d0.safe_hi;
  d.V = V;
  d.P = pl.P;
  d.chunk_elems = pl.chunk_elems;
  d.B = B;
  const int64_t items = static_cast<int64_t>(B) * pl.P;
  const int64_t g = static_cast<int64_t>(sm_count()) * kK3CtasPerSm;
  d.G = static_cast<int32_t>(items < g ? items : g);
  d.c = c;
  d.draws = reinterpret_cast<const DrawDesc*>(w + pl.off_draw);
  d.excl = reinterpret_cast<const int32_t*>(w + pl.off_excl);
  d.excl_stride = pl.excl_stride;
  d.part = reinterpret_cast<float2*>(w + pl.off_k3part);
  d.out_cols = out_cols;
  d.out_tokens = out_tokens;
  d.out_logprob = out_logprob;
  d.out_mu = out_mu;
  d.out_nodes = nullptr;
  d.out_status = nullptr;
  d.fin_here = 0;
  return d;
}

// Draft-tree construction's row pass (a TMA ring of kTbSmemBytes per CTA).
template <int ES>
cudaError_t launch_row_topk(const RowTopkArgs& a, int grid, cudaStream_t stream) {
  const cudaError_t e = once_per_device(kAttrRowTopk << (ES == 2 ? 0 : 8),
                                        [] { return set_smem_attrs(row_topk_kernel<ES>, kTbSmemBytes); });
  if (e != cudaSuccess) return e;
  return launch(row_topk_kernel<ES>, grid, kTbThreads, kTbSmemBytes, stream, true, a);
}

// The draw: chunk sums over the drawn rows (K3a), then the pick (K3b).
template <int ES>
cudaError_t launch_draw(const DrawArgs& d, cudaStream_t stream) {
  cudaError_t e = once_per_device(kAttrDraw << (ES == 2 ? 0 : 8),
                                  [] { return set_smem_attrs(draw_sum_kernel<ES>, kK3SmemBytes); });
  if (e != cudaSuccess) return e;
  e = launch(draw_sum_kernel<ES>, d.G, kK3Threads, kK3SmemBytes, stream, true, d);
  if (e != cudaSuccess) return e;
  return launch(draw_pick_kernel<ES>, d.B, kK3PickThreads, 0, stream, true, d);
}

// Stochastic tree call: merge, walk and draw in one cluster kernel (one
// cluster of kTwCluster CTAs per request).
template <int ES>
cudaError_t launch_tree_walk_draw(const TwArgs& w, cudaStream_t stream) {
  const cudaError_t e = once_per_device(kAttrTreeDraw << (ES == 2 ? 0 : 8), [] {
    return set_smem_attrs(tree_walk_draw_kernel<ES>, static_cast<int>(tw_layout(kMaxTreeNodes, kTwMaxChunks).total));
  });
  if (e != cudaSuccess) return e;
  return launch(tree_walk_draw_kernel<ES>, w.t.B * kTwCluster, kTwThreads, tw_layout(w.t.N, w.nch).total, stream,
                true, w);
}

// Finish-step arguments of a call (disabled when fin is null).
sv_status finish_args(const sv_finish_params* fin, int32_t offered, FinishArgs* f) {
  std::memset(f, 0, sizeof(*f));
  if (!fin) return SV_OK;
  if (!fin->out_len || !aligned(fin->out_len, 4)) return SV_ERR_INVALID_ARG;
  if (fin->n_stop < 0 || fin->n_stop > SV_MAX_STOP_IDS || (fin->n_stop > 0 && !fin->stop_ids)) return SV_ERR_INVALID_ARG;
  if (!aligned(fin->stop_ids, 4) || !aligned(fin->max_new, 4) || !aligned(fin->counters, 8)) return SV_ERR_INVALID_ARG;
  f->stop_ids = fin->stop_ids;
  f->n_stop = fin->n_stop;
  f->max_new = fin->max_new;
  f->out_len = fin->out_len;
  f->counters = reinterpret_cast<long long*>(fin->counters);
  f->offered = offered;
  return SV_OK;
}

bool outputs_aligned(const void* a, const void* b, const void* c, const void* d, const void* e) {
  return aligned(a, 4) && aligned(b, 4) && aligned(c, 4) && aligned(d, 4) && aligned(e, 4);
}

}  // namespace

extern "C" {

int32_t spec_verify_abi_version(void) { return SPEC_VERIFY_ABI_VERSION; }

const char* spec_verify_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "SV_OK: success";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: a pointer, size, stride or parameter is invalid";
    case SV_ERR_UNSUPPORTED_DTYPE: return "SV_ERR_UNSUPPORTED_DTYPE: dtype must be SV_F32 or SV_BF16";
    case SV_ERR_WORKSPACE_TOO_SMALL: return "SV_ERR_WORKSPACE_TOO_SMALL: workspace_bytes is below the required size";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA launch failed";
    case SV_ERR_NOT_SUPPORTED: return "SV_ERR_NOT_SUPPORTED: valid request not implemented by this build";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded wait inside a kernel gave up (SV_STATUS_TIMEOUT)";
    default: return "unknown sv_status";
  }
}

size_t spec_verify_greedy_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype) {
  Plan pl;
  if (B < 0 || K < 0 || !make_plan(static_cast<int64_t>(B) * (K + 1), 0, B, V, elem_size(dtype), false, 0, 0, &pl))
    return 0;
  return pl.total;
}

size_t spec_verify_sample_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype,
                                         int32_t has_draft_logits) {
  Plan pl;
  const int64_t rd = has_draft_logits ? static_cast<int64_t>(B) * K : 0;
  if (B < 0 || K < 0 ||
      !make_plan(static_cast<int64_t>(B) * (K + 1), rd, B, V, elem_size(dtype), true, 1, rd, &pl))
    return 0;
  return pl.total;
}

size_t spec_verify_tree_workspace_size(int32_t B, int32_t N, int32_t V, int32_t dtype) {
  Plan pl;
  if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES ||
      !make_plan(static_cast<int64_t>(B) * N, 0, B, V, elem_size(dtype), true, N, 0, &pl))
    return 0;
  return pl.total;
}

size_t spec_verify_workspace_size(int32_t B, int32_t rows_per_req, int32_t V, int32_t dtype) {
  if (B < 0 || rows_per_req < 1 || V < 1 || elem_size(dtype) == 0) return 0;
  const int32_t K = rows_per_req - 1;
  size_t need = spec_verify_greedy_workspace_size(B, K, V, dtype);
  const size_t with_draft = spec_verify_sample_workspace_size(B, K, V, dtype, 1);
  const size_t without = spec_verify_sample_workspace_size(B, K, V, dtype, 0);
  if (need == 0 || with_draft == 0 || without == 0) return 0;
  need = need > with_draft ? need : with_draft;
  need = need > without ? need : without;
  if (rows_per_req <= SV_MAX_TREE_NODES) {
    const size_t tree = spec_verify_tree_workspace_size(B, rows_per_req, V, dtype);
    if (tree == 0) return 0;
    need = need > tree ? need : tree;
  }
  return need;
}

sv_status spec_verify_check_status(const int32_t* status_host, int32_t B) {
  if (B < 0 || (B > 0 && !status_host)) return SV_ERR_INVALID_ARG;
  for (int32_t b = 0; b < B; ++b)
    if (status_host[b] & SV_STATUS_TIMEOUT) return SV_ERR_TIMEOUT;
  return SV_OK;
}

sv_status spec_verify_selftest_wait(int32_t* out_status, void* stream) {
  if (!out_status || !aligned(out_status, 4)) return SV_ERR_INVALID_ARG;
  const cudaError_t e = launch(selftest_wait_kernel, 1, 32, 0, static_cast<cudaStream_t>(stream), false, out_status);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify_greedy(const void* target_logits, int32_t dtype, int64_t row_stride,
                             const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                             int32_t* out_tokens, int32_t* out_num_accepted, float* out_logprob,
                             float* out_mu, int32_t* out_status, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return spec_verify_greedy_ex(target_logits, dtype, row_stride, draft_tokens, B, K, V, out_tokens,
                               out_num_accepted, out_logprob, out_mu, out_status, nullptr, workspace,
                               workspace_bytes, stream);
}

sv_status spec_verify_greedy_ex(const void* target_logits, int32_t dtype, int64_t row_stride,
                                const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                int32_t* out_tokens, int32_t* out_num_accepted, float* out_logprob,
                                float* out_mu, int32_t* out_status, const sv_finish_params* finish,
                                void* workspace, size_t workspace_bytes, void* stream) {
  const int es = elem_size(dtype);
  if (es == 0) return SV_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || K < 0 || V < 1 || row_stride < V) return SV_ERR_INVALID_ARG;
  FinishArgs fa;
  if (finish_args(finish, K, &fa) != SV_OK) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || (K > 0 && !draft_tokens) || !out_tokens || !out_num_accepted || !workspace)
    return SV_ERR_INVALID_ARG;
  if (!aligned(target_logits, es) || !aligned(workspace, 16) || !aligned(draft_tokens, 4) ||
      !outputs_aligned(out_tokens, out_num_accepted, out_logprob, out_mu, out_status))
    return SV_ERR_INVALID_ARG;
  Plan pl;
  const int64_t rows = static_cast<int64_t>(B) * (K + 1);
  if (!make_plan(rows, 0, B, V, es, false, 0, 0, &pl)) return SV_ERR_INVALID_ARG;
  if (workspace_bytes < pl.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float c = kLog2e;
  const RowStatsArgs r = row_stats_args(pl, target_logits, row_stride, rows, nullptr, 0, 0, V, es, c, workspace);
  cudaError_t e = es == 2 ? launch_row_stats<2>(r, st) : launch_row_stats<4>(r, st);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  ChainArgs a;
  std::memset(&a, 0, sizeof(a));
  a.tgt = static_cast<const uint8_t*>(target_logits);
  a.tgt_stride = row_stride * es;
  a.drafts = draft_tokens;
  a.B = B;
  a.K = K;
  a.V = V;
  a.part = r.partials;
  a.T = r.T;
  a.G = r.G;
  a.c = c;
  a.greedy = 1;
  a.fin = fa;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.out_logprob = out_logprob;
  a.out_mu = out_mu;
  a.out_status = out_status;
  // Rows that span more than ~3.5 row-pass CTAs (small batches) have more
  // partials than one round trip of two loads per lane covers.
  const bool wide = static_cast<double>(V) * r.G > 3.5 * static_cast<double>(r.T);
  if (wide)
    e = es == 2 ? launch(chain_decide_kernel<2, kK2MinBlocksGreedy, true>, B, kK2Threads, 0, st, true, a)
                : launch(chain_decide_kernel<4, kK2MinBlocksGreedy, true>, B, kK2Threads, 0, st, true, a);
  else
    e = es == 2 ? launch(chain_decide_kernel<2, kK2MinBlocksGreedy>, B, kK2Threads, 0, st, true, a)
                : launch(chain_decide_kernel<4, kK2MinBlocksGreedy>, B, kK2Threads, 0, st, true, a);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify_sample(const void* target_logits, int32_t dtype, int64_t row_stride,
                             const void* draft_logits, int64_t draft_row_stride,
                             const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                             float temperature, const float* uniforms, sv_rule_params rule,
                             int32_t* out_tokens, int32_t* out_num_accepted, float* out_logprob,
                             float* out_mu, int32_t* out_status, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return spec_verify_sample_ex(target_logits, dtype, row_stride, draft_logits, draft_row_stride,
                               draft_tokens, B, K, V, temperature, uniforms, rule, out_tokens,
                               out_num_accepted, out_logprob, out_mu, out_status, nullptr, workspace,
                               workspace_bytes, stream);
}

sv_status spec_verify_sample_ex(const void* target_logits, int32_t dtype, int64_t row_stride,
                                const void* draft_logits, int64_t draft_row_stride,
                                const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                float temperature, const float* uniforms, sv_rule_params rule,
                                int32_t* out_tokens, int32_t* out_num_accepted, float* out_logprob,
                                float* out_mu, int32_t* out_status, const sv_finish_params* finish,
                                void* workspace, size_t workspace_bytes, void* stream) {
  const int es = elem_size(dtype);
  if (es == 0) return SV_ERR_UNSUPPORTED_DTYPE;
  FinishArgs fa;
  if (finish_args(finish, K, &fa) != SV_OK) return SV_ERR_INVALID_ARG;
  if (B < 0 || K < 0 || V < 1 || row_stride < V) return SV_ERR_INVALID_ARG;
  if (draft_logits && draft_row_stride < V) return SV_ERR_INVALID_ARG;
  if (!valid_temperature(temperature)) return SV_ERR_INVALID_ARG;
  const sv_status rs = check_rule(rule);
  if (rs != SV_OK) return rs;
  if (B == 0) return SV_OK;
  if (!target_logits || (K > 0 && !draft_tokens) || !uniforms || !out_tokens || !out_num_accepted ||
      !workspace)
    return SV_ERR_INVALID_ARG;
  if (!aligned(target_logits, es) || (draft_logits && !aligned(draft_logits, es)) ||
      !aligned(workspace, 16) || !aligned(draft_tokens, 4) || !aligned(uniforms, 4) ||
      !outputs_aligned(out_tokens, out_num_accepted, out_logprob, out_mu, out_status))
    return SV_ERR_INVALID_ARG;
  Plan pl;
  const int64_t rows_t = static_cast<int64_t>(B) * (K + 1);
  const int64_t rows_d = draft_logits ? static_cast<int64_t>(B) * K : 0;
  if (!make_plan(rows_t, rows_d, B, V, es, true, 1, rows_d, &pl)) return SV_ERR_INVALID_ARG;
  if (workspace_bytes < pl.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float c = kLog2e / temperature;
  RowStatsArgs r = row_stats_args(pl, target_logits, row_stride, rows_t, draft_logits, draft_row_stride, rows_d,
                                  V, es, c, workspace);
  cudaError_t e = es == 2 ? launch_row_stats<2>(r, st) : launch_row_stats<4>(r, st);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  ChainArgs a;
  std::memset(&a, 0, sizeof(a));
  a.tgt = static_cast<const uint8_t*>(target_logits);
  a.tgt_stride = row_stride * es;
  a.dft = static_cast<const uint8_t*>(draft_logits);
  a.dft_stride = draft_logits ? draft_row_stride * es : 0;
  a.drafts = draft_tokens;
  a.uniforms = uniforms;
  a.B = B;
  a.K = K;
  a.V = V;
  a.part = r.partials;
  a.T = r.T;
  a.G = r.G;
  a.c = c;
  a.greedy = 0;
  a.rule = rule_args(rule);
  if (a.rule.top_k > 0 && K > 0) {
    float* thr = reinterpret_cast<float*>(w + pl.off_thr);
    e = launch_topk(target_logits, row_stride * es, K, K + 1, V, a.rule.top_k, nullptr, thr, B * K, es, st);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    a.rule.thr = thr;
  }
  const bool mu_pass = draft_logits && a.rule.rule != SV_RULE_EXACT && K > 0;
  a.mu_counters = mu_pass ? reinterpret_cast<uint32_t*>(w + pl.off_mucnt) : nullptr;
  DrawArgs d = draw_args(pl, target_logits, row_stride, rows_t, draft_logits, draft_logits ? draft_row_stride : 0,
                         rows_d, B, V, es, c, workspace, K + 1, out_tokens, out_logprob, out_mu);
  // The exact rule with draft logits and short chains decides inside the
  // draw's chunk-sum kernel (no decide kernel), when no chunk-sum CTA's item
  // range spans more requests than it decides.
  const int64_t items_per_cta = (static_cast<int64_t>(B) * pl.P + d.G - 1) / d.G;
  const bool fuse = draft_logits && a.rule.rule == SV_RULE_EXACT && a.rule.top_k == 0 && K + 1 <= kFusedMaxRows &&
                    (items_per_cta + pl.P - 1) / pl.P + 1 <= kK3Req;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.out_logprob = out_logprob;
  a.out_mu = out_mu;
  a.out_status = out_status;
  a.draws = reinterpret_cast<DrawDesc*>(w + pl.off_draw);
  a.excl = reinterpret_cast<int32_t*>(w + pl.off_excl);
  a.excl_stride = pl.excl_stride;
  if (fuse) {
    d.fused = 1;
    d.k1_part = r.partials;
    d.k1_T = r.T;
    d.k1_G = r.G;
    d.K = K;
    d.drafts = draft_tokens;
    d.uniforms = uniforms;
    d.out_num = out_num_accepted;
    d.draws_out = a.draws;
  } else {
    e = es == 2 ? launch(chain_decide_kernel<2, kK2MinBlocksDraw>, B, kK2Threads, 0, st, true, a)
                : launch(chain_decide_kernel<4, kK2MinBlocksDraw>, B, kK2Threads, 0, st, true, a);
    if (e != cudaSuccess) return SV_ERR_CUDA;
  }
  d.out_status = out_status;
  d.fin = fa;
  d.fin_here = (fa.out_len && !mu_pass) ? 1 : 0;
  e = es == 2 ? launch_draw<2>(d, st) : launch_draw<4>(d, st);
  if (e != cudaSuccess || !mu_pass) return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
  MuArgs m;
  std::memset(&m, 0, sizeof(m));
  m.tgt = a.tgt;
  m.tgt_stride = a.tgt_stride;
  m.dft = a.dft;
  m.dft_stride = a.dft_stride;
  m.drafts = draft_tokens;
  m.B = B;
  m.K = K;
  m.V = V;
  m.P = pl.P;
  m.chunk_elems = pl.chunk_elems;
  m.part = r.partials;
  m.T = r.T;
  m.G = r.G;
  m.c = c;
  m.rule = a.rule;
  m.num = out_num_accepted;
  m.tokens = out_tokens;
  m.out_mu = out_mu;
  m.out_tokens = out_tokens;
  m.out_logprob = out_logprob;
  m.out_status = out_status;
  m.fin = fa;
  m.mpart = reinterpret_cast<float2*>(w + pl.off_mupart);
  m.counters = a.mu_counters;
  const int grid_mu = B * K * pl.P;
  e = es == 2 ? launch(mu_pass_kernel<2>, grid_mu, kMuThreads, 0, st, true, m)
              : launch(mu_pass_kernel<4>, grid_mu, kMuThreads, 0, st, true, m);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify_tree(const void* target_logits, int32_t dtype, int64_t row_stride,
                           const int32_t* node_tokens, const int32_t* parents, int32_t B,
                           int32_t N, int32_t V, int32_t max_depth, float temperature,
                           const float* uniforms, sv_rule_params rule, int32_t* out_tokens,
                           int32_t* out_nodes, int32_t* out_num_accepted, float* out_logprob,
                           float* out_mu, int32_t* out_status, void* workspace,
                           size_t workspace_bytes, void* stream) {
  return spec_verify_tree_ex(target_logits, dtype, row_stride, node_tokens, parents, B, N, V, max_depth,
                             temperature, uniforms, rule, out_tokens, out_nodes, out_num_accepted,
                             out_logprob, out_mu, out_status, nullptr, workspace, workspace_bytes, stream);
}

sv_status spec_verify_tree_ex(const void* target_logits, int32_t dtype, int64_t row_stride,
                              const int32_t* node_tokens, const int32_t* parents, int32_t B,
                              int32_t N, int32_t V, int32_t max_depth, float temperature,
                              const float* uniforms, sv_rule_params rule, int32_t* out_tokens,
                              int32_t* out_nodes, int32_t* out_num_accepted, float* out_logprob,
                              float* out_mu, int32_t* out_status, const sv_finish_params* finish,
                              void* workspace, size_t workspace_bytes, void* stream) {
  const int es = elem_size(dtype);
  if (es == 0) return SV_ERR_UNSUPPORTED_DTYPE;
  FinishArgs fa;
  if (finish_args(finish, max_depth, &fa) != SV_OK) return SV_ERR_INVALID_ARG;
  if (B < 0 || N < 1 || N > SV_MAX_TREE_NODES || V < 1 || row_stride < V || max_depth < 0 ||
      max_depth > INT32_MAX - 1)
    return SV_ERR_INVALID_ARG;
  const bool greedy = temperature == 0.f;
  if (!greedy && !valid_temperature(temperature)) return SV_ERR_INVALID_ARG;
  if (!greedy) {
    const sv_status rs = check_rule(rule);
    if (rs != SV_OK) return rs;
  }
  if (B == 0) return SV_OK;
  if (!target_logits || !node_tokens || !parents || (!greedy && !uniforms) || !out_tokens ||
      !out_nodes || !out_num_accepted || !workspace)
    return SV_ERR_INVALID_ARG;
  if (!aligned(target_logits, es) || !aligned(workspace, 16) || !aligned(node_tokens, 4) ||
      !aligned(parents, 4) || !aligned(uniforms, 4) || !aligned(out_nodes, 4) ||
      !outputs_aligned(out_tokens, out_num_accepted, out_logprob, out_mu, out_status))
    return SV_ERR_INVALID_ARG;
  Plan pl;
  const int64_t rows = static_cast<int64_t>(B) * N;
  if (!make_plan(rows, 0, B, V, es, true, N, 0, &pl)) return SV_ERR_INVALID_ARG;
  if (workspace_bytes < pl.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float c = greedy ? kLog2e : kLog2e / temperature;
  const RowStatsArgs r = row_stats_args(pl, target_logits, row_stride, rows, nullptr, 0, 0, V, es, c, workspace);
  cudaError_t e = es == 2 ? launch_row_stats<2>(r, st) : launch_row_stats<4>(r, st);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  TreeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.tgt = static_cast<const uint8_t*>(target_logits);
  a.tgt_stride = row_stride * es;
  a.tokens = node_tokens;
  a.parents = parents;
  a.uniforms = uniforms;
  a.B = B;
  a.N = N;
  a.V = V;
  a.max_depth = max_depth;
  a.part = r.partials;
  a.T = r.T;
  a.G = r.G;
  a.c = c;
  a.greedy = greedy ? 1 : 0;
  a.fin = fa;
  a.rule = rule_args(rule);
  if (!greedy && a.rule.top_k > 0) {
    float* thr = reinterpret_cast<float*>(w + pl.off_thr);
    e = launch_topk(target_logits, row_stride * es, N, N, V, a.rule.top_k, parents, thr, B * N, es, st);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    a.rule.thr = thr;
  }
  a.out_tokens = out_tokens;
  a.out_nodes = out_nodes;
  a.out_num = out_num_accepted;
  a.out_logprob = out_logprob;
  a.out_mu = out_mu;
  a.out_status = out_status;
  a.draws = reinterpret_cast<DrawDesc*>(w + pl.off_draw);
  a.excl = reinterpret_cast<int32_t*>(w + pl.off_excl);
  a.excl_stride = pl.excl_stride;
  // One kernel for the stochastic walk and its draw when every chunk of a
  // row starts on a 16-byte boundary and a row's chunks fit the cluster.
  if (!greedy && aligned(target_logits, 16) && (row_stride * es) % 16 == 0 && pl.P <= kTwMaxP) {
    TwArgs tw;
    std::memset(&tw, 0, sizeof(tw));
    tw.t = a;
    tw.tgt_hi = row_set(target_logits, row_stride, rows, V, es).safe_hi;
    tw.P = pl.P;
    tw.chunk_elems = pl.chunk_elems;
    tw.nch = (pl.P + kTwCluster - 1) / kTwCluster;
    e = es == 2 ? launch_tree_walk_draw<2>(tw, st) : launch_tree_walk_draw<4>(tw, st);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
  }
  e = es == 2 ? launch(tree_decide_kernel<2>, B, kK2Threads, 0, st, true, a)
              : launch(tree_decide_kernel<4>, B, kK2Threads, 0, st, true, a);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  if (greedy) return SV_OK;
  DrawArgs d = draw_args(pl, target_logits, row_stride, rows, nullptr, 0, 0, B, V, es, c, workspace, max_depth + 1,
                         out_tokens, out_logprob, out_mu);
  d.out_nodes = out_nodes;
  d.out_status = out_status;
  d.fin = fa;
  d.fin_here = fa.out_len ? 1 : 0;
  e = es == 2 ? launch_draw<2>(d, st) : launch_draw<4>(d, st);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

size_t spec_tree_build_workspace_size(int32_t B, int32_t depth, int32_t topk, int32_t V) {
  if (B < 0 || depth < 1 || topk < 1 || topk > kTbMaxK || V < 1) return 0;
  const int64_t P = (V + kTbPieceElems - 1) / kTbPieceElems;
  const int64_t rows = static_cast<int64_t>(B) * (1 + static_cast<int64_t>(depth - 1) * topk);
  return align_up(static_cast<size_t>(rows > 0 ? rows * P : 1) * sizeof(TopRow), kAlign);
}

sv_status spec_tree_build(const void* draft_logits, int32_t dtype, int64_t row_stride, int32_t B, int32_t V,
                          int32_t depth, int32_t topk, int32_t n_nodes, float temperature,
                          int32_t* out_tokens, int32_t* out_parents, float* out_scores, int32_t* out_status,
                          void* workspace, size_t workspace_bytes, void* stream) {
  const int es = elem_size(dtype);
  if (es == 0) return SV_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || V < 1 || row_stride < V || depth < 1 || topk < 1 || topk > kTbMaxK || topk > V)
    return SV_ERR_INVALID_ARG;
  const int64_t cands = topk + static_cast<int64_t>(depth - 1) * topk * topk;
  if (cands > kTbMaxCands || n_nodes < 1 || n_nodes > 1 + cands || n_nodes > SV_MAX_TREE_NODES)
    return SV_ERR_INVALID_ARG;
  if (!valid_temperature(temperature)) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!draft_logits || !out_tokens || !out_parents || !workspace) return SV_ERR_INVALID_ARG;
  if (!aligned(draft_logits, es) || !aligned(workspace, 16) || !aligned(out_tokens, 4) || !aligned(out_parents, 4) ||
      !aligned(out_scores, 4) || !aligned(out_status, 4))
    return SV_ERR_INVALID_ARG;
  const int32_t R = 1 + (depth - 1) * topk;
  if (R > kTbMaxRows) return SV_ERR_INVALID_ARG;
  const int64_t rows = static_cast<int64_t>(B) * R;
  if (rows > INT32_MAX) return SV_ERR_INVALID_ARG;
  if (workspace_bytes < spec_tree_build_workspace_size(B, depth, topk, V)) return SV_ERR_WORKSPACE_TOO_SMALL;
  const int32_t P = (V + kTbPieceElems - 1) / kTbPieceElems;
  if (rows * P > INT32_MAX) return SV_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float c = kLog2e / temperature;
  RowTopkArgs ra;
  const RowSet rs = row_set(draft_logits, row_stride, rows, V, es);
  ra.base = rs.base;
  ra.stride_bytes = rs.stride_bytes;
  ra.safe_lo = rs.safe_lo;
  ra.safe_hi = rs.safe_hi;
  ra.V = V;
  ra.P = P;
  ra.c = c;
  ra.out = static_cast<TopRow*>(workspace);
  cudaError_t e = es == 2 ? launch_row_topk<2>(ra, static_cast<int>(rows * P), st)
                          : launch_row_topk<4>(ra, static_cast<int>(rows * P), st);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  TreeSelectArgs ta;
  ta.rows = ra.out;
  ta.R = R;
  ta.P = P;
  ta.depth = depth;
  ta.topk = topk;
  ta.n_nodes = n_nodes;
  ta.c = c;
  ta.out_tokens = out_tokens;
  ta.out_parents = out_parents;
  ta.out_scores = out_scores;
  ta.out_status = out_status;
  e = launch(tree_select_kernel, B, kTbSelThreads, 0, st, true, ta);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_kv_compact(void* kv, int64_t token_stride_bytes, int32_t row_bytes, const int32_t* page_table,
                          int32_t max_pages, int32_t page_size, const int32_t* seq_base, const int32_t* path_nodes,
                          int32_t path_cols, const int32_t* num_accepted, int32_t B, int32_t max_nodes,
                          int32_t* out_len, int32_t* out_status, void* stream) {
  if (B < 0 || row_bytes < 16 || row_bytes % 16 != 0 || token_stride_bytes < row_bytes || token_stride_bytes % 16 != 0 ||
      max_pages < 1 || page_size < 1 || path_cols < 1 || max_nodes < 1)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!kv || !page_table || !seq_base || !path_nodes || !num_accepted || !out_len) return SV_ERR_INVALID_ARG;
  if (!aligned(kv, 16) || !aligned(page_table, 4) || !aligned(seq_base, 4) || !aligned(path_nodes, 4) ||
      !aligned(num_accepted, 4) || !aligned(out_len, 4) || !aligned(out_status, 4))
    return SV_ERR_INVALID_ARG;
  KvCompactArgs k;
  k.kv = static_cast<uint8_t*>(kv);
  k.token_stride = token_stride_bytes;
  k.page_bytes = static_cast<int64_t>(page_size) * token_stride_bytes;
  k.row_bytes = row_bytes;
  k.page_table = page_table;
  k.max_pages = max_pages;
  k.page_size = page_size;
  k.seq_base = seq_base;
  k.path_nodes = path_nodes;
  k.path_cols = path_cols;
  k.num_accepted = num_accepted;
  k.max_nodes = max_nodes;
  k.chunks = (row_bytes + kKvChunkBytes - 1) / kKvChunkBytes;
  k.out_len = out_len;
  k.out_status = out_status;
  const int64_t grid = static_cast<int64_t>(B) * k.chunks;
  if (grid > INT32_MAX) return SV_ERR_INVALID_ARG;
  const cudaError_t e = launch(kv_compact_kernel, static_cast<int>(grid), kKvThreads, 0,
                               static_cast<cudaStream_t>(stream), true, k);
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify_greedy_early(const void* target_logits, int32_t dtype, int64_t row_stride,
                                   const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                   int32_t* out_tokens, int32_t* out_num_accepted, float* out_logprob,
                                   float* out_mu, int32_t* out_status, int32_t* state,
                                   uint64_t* out_bytes_read, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  const int es = elem_size(dtype);
  if (es == 0) return SV_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || K < 0 || V < 1 || row_stride < V) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || (K > 0 && !draft_tokens) || !out_tokens || !out_num_accepted || !workspace || !state)
    return SV_ERR_INVALID_ARG;
  if (!aligned(target_logits, es) || !aligned(workspace, 16) || !aligned(draft_tokens, 4) || !aligned(state, 4) ||
      !aligned(out_bytes_read, 8) || !outputs_aligned(out_tokens, out_num_accepted, out_logprob, out_mu, out_status))
    return SV_ERR_INVALID_ARG;
  Plan pl;
  const int64_t rows = static_cast<int64_t>(B) * (K + 1);
  if (!make_plan(rows, 0, B, V, es, false, 0, 0, &pl)) return SV_ERR_INVALID_ARG;
  if (workspace_bytes < pl.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float c = kLog2e;
  EarlyArgs e;
  e.rs = row_stats_args(pl, target_logits, row_stride, rows, nullptr, 0, 0, V, es, c, workspace);
  int64_t g = static_cast<int64_t>(sm_count()) * kK1CtasPerSm;
  if (g > rows) g = rows;
  if (g > kK1MaxCtas) g = kK1MaxCtas;
  e.rs.G = static_cast<int32_t>(g);
  e.B = B;
  e.R = K + 1;
  e.drafts = draft_tokens;
  e.state = state;
  e.done = state + B;
  // one partial per row at slot `row`; the spare kK1MaxCtas slots after them hold the CTAs' byte counts
  e.cta_bytes = reinterpret_cast<unsigned long long*>(e.rs.partials + rows);
  cudaError_t err = es == 2 ? launch_row_stats_early<2>(e, st) : launch_row_stats_early<4>(e, st);
  if (err != cudaSuccess) return SV_ERR_CUDA;
  ChainArgs a;
  std::memset(&a, 0, sizeof(a));
  a.tgt = static_cast<const uint8_t*>(target_logits);
  a.tgt_stride = row_stride * es;
  a.drafts = draft_tokens;
  a.B = B;
  a.K = K;
  a.V = V;
  a.part = e.rs.partials;
  a.T = e.rs.T;
  a.G = e.rs.G;
  a.c = c;
  a.greedy = 1;
  a.out_tokens = out_tokens;
  a.out_num = out_num_accepted;
  a.out_logprob = out_logprob;
  a.out_mu = out_mu;
  a.out_status = out_status;
  a.row_partials = 1;
  a.early_state = state;
  a.cta_bytes = e.cta_bytes;
  a.n_cta = e.rs.G;
  a.out_bytes = reinterpret_cast<unsigned long long*>(out_bytes_read);
  err = es == 2 ? launch(chain_decide_kernel<2, kK2MinBlocksGreedy>, B, kK2Threads, 0, st, true, a)
                : launch(chain_decide_kernel<4, kK2MinBlocksGreedy>, B, kK2Threads, 0, st, true, a);
  return err == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// ------------------------------------------------- no-allocation variant
//
// Scratch for spec_verify_greedy_static: a file-scope device array, so a
// caller that cannot allocate device memory still gets the workspace the
// greedy kernels need. Every GPU that loads the library holds one copy until
// the process exits. Host code must not pass g_static_scratch itself to a
// kernel (in host code that name is a host-side stand-in, not a device
// address); the device address is looked up once per device below.
static __device__ __align__(256) unsigned char g_static_scratch[SV_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_static_scratch_mu;
void* g_static_scratch_dev[64] = {nullptr};
}  // namespace

sv_status spec_verify_greedy_static(const void* target_logits, int32_t dtype, int64_t row_stride,
                                    const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                    int32_t* out_tokens, int32_t* out_num_accepted, float* out_logprob,
                                    float* out_mu, int32_t* out_status, void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (g_static_scratch_dev[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return SV_ERR_CUDA;
      g_static_scratch_dev[dev] = p;
    }
    scratch = g_static_scratch_dev[dev];
  }
  // The greedy path's own size check turns a request that needs more than
  // the static array into SV_ERR_WORKSPACE_TOO_SMALL before any launch.
  return spec_verify_greedy(target_logits, dtype, row_stride, draft_tokens, B, K, V, out_tokens,
                            out_num_accepted, out_logprob, out_mu, out_status, scratch,
                            SV_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"

// ------------------------------------------------- host-resident logits
//
// spec_verify_greedy_host: two device staging slots, a copy stream per
// device (created on first use, kept for the life of the process), and per
// group of requests: copy (copy stream) -> verify -> outputs back (caller's
// stream), with the next group's copy enqueued before this group's outputs
// so the copy engine never waits on the host.
namespace {
cudaStream_t g_copy_stream[kMaxDevices] = {nullptr};

cudaStream_t host_copy_stream() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_cache_mu);
  if (!g_copy_stream[dev]) {
    cudaStream_t s = nullptr;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    g_copy_stream[dev] = s;
  }
  return g_copy_stream[dev];
}

constexpr size_t kHostAlign = 256;

struct HostPlan {
  int32_t g = 0;   // requests per group
  size_t slot = 0, off_slot[2] = {0, 0}, off_drafts = 0, off_tok = 0, off_num = 0, off_lp = 0, off_mu = 0,
         off_st = 0, off_ws = 0, ws_bytes = 0, total = 0;
};

// Device layout of the host-path workspace: the staging slots hold rows
// packed at stride V.
bool host_plan(int32_t B, int32_t K, int32_t V, int32_t dtype, int32_t group, HostPlan* hp) {
  const int es = elem_size(dtype);
  if (es == 0 || B < 0 || K < 0 || V < 1 || group < 0) return false;
  const int64_t R = static_cast<int64_t>(K) + 1;
  const int64_t req_bytes = R * V * es;
  int64_t g = group > 0 ? group : static_cast<int64_t>(SV_HOST_GROUP_BYTES) / req_bytes;
  if (g < 1) g = 1;
  if (g > B) g = B > 0 ? B : 1;
  hp->g = static_cast<int32_t>(g);
  hp->ws_bytes = spec_verify_greedy_workspace_size(hp->g, K, V, dtype);
  if (hp->ws_bytes == 0) return false;
  size_t o = 0;
  hp->slot = align_up(static_cast<size_t>(g * req_bytes), kHostAlign);
  hp->off_slot[0] = o;
  o += hp->slot;
  hp->off_slot[1] = o;
  o += hp->slot;
  hp->off_drafts = o;
  o += align_up(static_cast<size_t>(B) * K * 4, kHostAlign);
  hp->off_tok = o;
  o += align_up(static_cast<size_t>(B * R) * 4, kHostAlign);
  hp->off_num = o;
  o += align_up(static_cast<size_t>(B) * 4, kHostAlign);
  hp->off_lp = o;
  o += align_up(static_cast<size_t>(B * R) * 4, kHostAlign);
  hp->off_mu = o;
  o += align_up(static_cast<size_t>(B * R) * 4, kHostAlign);
  hp->off_st = o;
  o += align_up(static_cast<size_t>(B) * 4, kHostAlign);
  hp->off_ws = o;
  o += align_up(hp->ws_bytes, kHostAlign);
  hp->total = o;
  return true;
}
}  // namespace

extern "C" {

size_t spec_verify_greedy_host_workspace_size(int32_t B, int32_t K, int32_t V, int32_t dtype, int32_t group) {
  HostPlan hp;
  return host_plan(B, K, V, dtype, group, &hp) ? hp.total : 0;
}

sv_status spec_verify_greedy_host(const void* target_logits, int32_t dtype, int64_t row_stride,
                                  const int32_t* draft_tokens, int32_t B, int32_t K, int32_t V,
                                  int32_t group, int32_t* out_tokens, int32_t* out_num_accepted,
                                  float* out_logprob, float* out_mu, int32_t* out_status,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const int es = elem_size(dtype);
  if (es == 0) return SV_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || K < 0 || V < 1 || row_stride < V || group < 0) return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!target_logits || (K > 0 && !draft_tokens) || !out_tokens || !out_num_accepted || !workspace)
    return SV_ERR_INVALID_ARG;
  if (!aligned(target_logits, es) || !aligned(workspace, kHostAlign) || !aligned(draft_tokens, 4) ||
      !outputs_aligned(out_tokens, out_num_accepted, out_logprob, out_mu, out_status))
    return SV_ERR_INVALID_ARG;
  HostPlan hp;
  if (!host_plan(B, K, V, dtype, group, &hp)) return SV_ERR_INVALID_ARG;
  if (workspace_bytes < hp.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t cs = host_copy_stream();
  if (!cs) return SV_ERR_CUDA;
  cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};   // start, ready[2], done[2]
  auto fail = [&]() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);   // released once pending work on it completes
    return SV_ERR_CUDA;
  };
  for (cudaEvent_t& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return fail();
  cudaEvent_t ev_start = ev[0], *ready = ev + 1, *done = ev + 3;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const int64_t R = static_cast<int64_t>(K) + 1;
  const int32_t* d_drafts = reinterpret_cast<const int32_t*>(w + hp.off_drafts);
  int32_t* d_tok = reinterpret_cast<int32_t*>(w + hp.off_tok);
  int32_t* d_num = reinterpret_cast<int32_t*>(w + hp.off_num);
  float* d_lp = reinterpret_cast<float*>(w + hp.off_lp);
  float* d_mu = reinterpret_cast<float*>(w + hp.off_mu);
  int32_t* d_st = reinterpret_cast<int32_t*>(w + hp.off_st);
  const int ngroups = static_cast<int>((static_cast<int64_t>(B) + hp.g - 1) / hp.g);
  const size_t row_bytes = static_cast<size_t>(V) * es;
  // The copy stream follows the work already on `stream` (earlier users of
  // the workspace).
  if (cudaEventRecord(ev_start, st) != cudaSuccess || cudaStreamWaitEvent(cs, ev_start, 0) != cudaSuccess)
    return fail();
  if (K > 0 && cudaMemcpyAsync(w + hp.off_drafts, draft_tokens, static_cast<size_t>(B) * K * 4,
                               cudaMemcpyHostToDevice, cs) != cudaSuccess)
    return fail();
  // Group i's logits into slot i % 2 once the verification of group i - 2
  // (the slot's last user) is done.
  auto copy_group = [&](int i) -> bool {
    const int s = i & 1;
    const int64_t b0 = static_cast<int64_t>(i) * hp.g;
    const int64_t gb = std::min<int64_t>(hp.g, B - b0);
    if (i >= 2 && cudaStreamWaitEvent(cs, done[s], 0) != cudaSuccess) return false;
    uint8_t* dst = w + hp.off_slot[s];
    const uint8_t* src = static_cast<const uint8_t*>(target_logits) + b0 * R * row_stride * es;
    cudaError_t e;
    if (row_stride == V)
      e = cudaMemcpyAsync(dst, src, static_cast<size_t>(gb * R) * row_bytes, cudaMemcpyHostToDevice, cs);
    else
      e = cudaMemcpy2DAsync(dst, row_bytes, src, static_cast<size_t>(row_stride) * es, row_bytes,
                            static_cast<size_t>(gb * R), cudaMemcpyHostToDevice, cs);
    return e == cudaSuccess && cudaEventRecord(ready[s], cs) == cudaSuccess;
  };
  if (!copy_group(0)) return fail();
  for (int i = 0; i < ngroups; ++i) {
    if (i + 1 < ngroups && !copy_group(i + 1)) return fail();
    const int s = i & 1;
    const int64_t b0 = static_cast<int64_t>(i) * hp.g;
    const int32_t gb = static_cast<int32_t>(std::min<int64_t>(hp.g, B - b0));
    if (cudaStreamWaitEvent(st, ready[s], 0) != cudaSuccess) return fail();
    const sv_status r = spec_verify_greedy(w + hp.off_slot[s], dtype, V, d_drafts + b0 * K, gb, K, V,
                                           d_tok + b0 * R, d_num + b0, d_lp + b0 * R, d_mu + b0 * R, d_st + b0,
                                           w + hp.off_ws, hp.ws_bytes, st);
    if (r != SV_OK) {
      fail();
      return r;
    }
    const size_t nrow = static_cast<size_t>(gb) * R * 4, nreq = static_cast<size_t>(gb) * 4;
    bool ok = cudaMemcpyAsync(out_tokens + b0 * R, d_tok + b0 * R, nrow, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
              cudaMemcpyAsync(out_num_accepted + b0, d_num + b0, nreq, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    if (ok && out_logprob)
      ok = cudaMemcpyAsync(out_logprob + b0 * R, d_lp + b0 * R, nrow, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    if (ok && out_mu) ok = cudaMemcpyAsync(out_mu + b0 * R, d_mu + b0 * R, nrow, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    if (ok && out_status)
      ok = cudaMemcpyAsync(out_status + b0, d_st + b0, nreq, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    if (!ok || cudaEventRecord(done[s], st) != cudaSuccess) return fail();
  }
  for (cudaEvent_t e : ev) cudaEventDestroy(e);
  return SV_OK;
}

}  // extern "C"
