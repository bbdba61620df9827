// lsx_api.cu -- the C ABI declared in include/lsx.h: argument validation,
// workspace sizing, dispatch to the kernels, the device status word and the
// host-side diagnostics.  Every check runs before any launch, so a call that
// returns an error has touched nothing.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "bwd_split.h"
#include "fwd_split.h"
#include "internal.h"
#include "ptx.cuh"

namespace lsx {

// One status word per device that loads the library.
__device__ int g_status_word;

namespace {

constexpr uint64_t kDefaultWaitNs = 10ull * 1000 * 1000 * 1000;  // 10 s
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_deterministic{0};

struct DevCache {
  bool ready = false;
  int sm_count = 0;
  int* status = nullptr;
};
std::mutex g_mu;
std::vector<DevCache> g_devs;

// ------------------------------------------------------- kernel timing
const char* const kKernelNames[kKidCount] = {
    "fwd_tc", "bwd_dkdv_tc", "bwd_dq_tc", "bwd_row_dot", "merge", "tree_merge",
    "decode_partials", "simt_fwd", "simt_bwd", "fill", "transpose", "block_lists",
    "bwd_fused_tc", "bwd_dq_convert"};
std::atomic<bool> g_timing{false};
struct TimedLaunch {
  int kid;
  cudaEvent_t a, b;
};
std::vector<TimedLaunch> g_launches;   // guarded by g_tmu
std::vector<cudaEvent_t> g_event_pool; // guarded by g_tmu
std::mutex g_tmu;
int g_open_kid = -1;
cudaEvent_t g_open_ev = nullptr;

cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

void timing_begin(int kid, cudaStream_t s) {
  if (!g_timing.load()) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  g_open_kid = kid;
  g_open_ev = pooled_event();
  cudaEventRecord(g_open_ev, s);
}

void timing_end(int kid, cudaStream_t s) {
  if (!g_timing.load()) return;
  std::lock_guard<std::mutex> lk(g_tmu);
  if (g_open_kid != kid || g_open_ev == nullptr) return;
  cudaEvent_t e = pooled_event();
  cudaEventRecord(e, s);
  g_launches.push_back({kid, g_open_ev, e});
  g_open_kid = -1;
  g_open_ev = nullptr;
}

namespace {
// ------------------------------------------------------- schedule trace
std::mutex g_trmu;
uint64_t* g_trace_buf = nullptr;  // caller's device buffer (words)
size_t g_trace_cap = 0;           // words
size_t g_trace_used = 0;          // words handed out since lsx_trace_enable
}  // namespace

uint64_t* trace_record(int kid, int64_t grid) {
  (void)kid;
  std::lock_guard<std::mutex> lk(g_trmu);
  if (g_trace_buf == nullptr) return nullptr;
  const size_t need = static_cast<size_t>(trace_words(grid));
  if (g_trace_used + need > g_trace_cap) return nullptr;
  uint64_t* rec = g_trace_buf + g_trace_used;
  g_trace_used += need;
  return rec;
}

int device_ctx(DeviceCtx* ctx) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LSX_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (static_cast<int>(g_devs.size()) <= dev) g_devs.resize(dev + 1);
  DevCache& dc = g_devs[dev];
  if (!dc.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return LSX_ERR_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return LSX_ERR_DEVICE;  // sm_103 only
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return LSX_ERR_DEVICE;
    dc.sm_count = prop.multiProcessorCount;
    dc.status = static_cast<int*>(addr);
    dc.ready = true;
  }
  ctx->device = dev;
  ctx->sm_count = dc.sm_count;
  ctx->status = dc.status;
  ctx->wait_ns = g_wait_ns.load();
  ctx->deterministic = g_deterministic.load();
  return LSX_OK;
}

namespace {

// ---------------------------------------------------------- validation
int check_view(const lsx_tensor* t) {
  if (t == nullptr) return LSX_ERR_NULL;
  if (t->data == nullptr && t->N != 0) return LSX_ERR_NULL;  // empty views may be NULL
  if (t->dtype != LSX_BF16 && t->dtype != LSX_F32) return LSX_ERR_DTYPE;
  if (t->B <= 0 || t->H <= 0 || t->N < 0 || t->D <= 0) return LSX_ERR_SHAPE;
  if (t->stride_b < 0 || t->stride_h < 0 || t->stride_n < 0) return LSX_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(t->data) % 16 != 0) return LSX_ERR_ALIGN;
  return LSX_OK;
}

int elem_size(int dtype) { return dtype == LSX_F32 ? 4 : 2; }

// A row of D elements is read/written with 16-byte vectors (or 8-byte for
// bf16 rows of 64/128 in the merge kernels): rows must start 16-B aligned.
int check_row_aligned(const lsx_tensor* t) {
  const int64_t vec = 16 / elem_size(t->dtype);
  if (t->stride_n % vec || t->stride_h % vec || t->stride_b % vec) return LSX_ERR_ALIGN;
  return LSX_OK;
}

int check_lse(const lsx_tensor* l, const lsx_tensor* like) {
  if (l == nullptr || l->data == nullptr) return LSX_ERR_NULL;
  if (l->dtype != LSX_F32) return LSX_ERR_DTYPE;
  if (l->D != 1 || l->B != like->B || l->H != like->H || l->N != like->N) return LSX_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(l->data) % 4 != 0) return LSX_ERR_ALIGN;
  if (l->stride_b < 0 || l->stride_h < 0 || l->stride_n < 0) return LSX_ERR_SHAPE;
  return LSX_OK;
}

bool same_bhn_d(const lsx_tensor* a, const lsx_tensor* b) {
  return a->B == b->B && a->H == b->H && a->N == b->N && a->D == b->D;
}

#define LSX_TRY(expr)          \
  do {                         \
    const int _rc = (expr);    \
    if (_rc != LSX_OK) return _rc; \
  } while (0)

// q [B,Hq,Lq,D], k/v [B,Hkv,Lk,D], same dtype, D in {64,128}, Hq % Hkv == 0.
int check_qkv(const lsx_tensor* q, const lsx_tensor* k, const lsx_tensor* v) {
  LSX_TRY(check_view(q));
  LSX_TRY(check_view(k));
  LSX_TRY(check_view(v));
  if (k->dtype != q->dtype || v->dtype != q->dtype) return LSX_ERR_DTYPE;
  if (k->B != q->B || v->B != q->B || k->D != q->D || v->D != q->D ||
      v->H != k->H || v->N != k->N)
    return LSX_ERR_SHAPE;
  if (q->H % k->H != 0) return LSX_ERR_SHAPE;
  if (q->D != 64 && q->D != 128) return LSX_ERR_UNSUPPORTED;
  LSX_TRY(check_row_aligned(q));
  LSX_TRY(check_row_aligned(k));
  LSX_TRY(check_row_aligned(v));
  // TMA: every coordinate must fit a 32-bit signed integer
  const int64_t lim = int64_t(1) << 31;
  if (q->N >= lim || k->N >= lim || q->H >= lim || q->B >= lim) return LSX_ERR_UNSUPPORTED;
  return LSX_OK;
}

float resolve_scale(float scale, int64_t d) {
  return scale > 0.f ? scale : 1.f / sqrtf(static_cast<float>(d));
}

cudaStream_t as_stream(lsx_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace
}  // namespace lsx

using namespace lsx;

extern "C" {

const char* lsx_version(void) { return "lsx 0.1 sm_103a"; }

const char* lsx_status_string(int code) {
  switch (code) {
    case LSX_OK: return "ok";
    case LSX_ERR_NULL: return "null pointer";
    case LSX_ERR_SHAPE: return "shape mismatch";
    case LSX_ERR_DTYPE: return "unsupported dtype combination";
    case LSX_ERR_ALIGN: return "misaligned base or stride";
    case LSX_ERR_UNSUPPORTED: return "unsupported size or option";
    case LSX_ERR_WORKSPACE: return "workspace missing or too small";
    case LSX_ERR_LAUNCH: return "CUDA launch or API failure";
    case LSX_ERR_TIMEOUT: return "device-side bounded wait ran out";
    case LSX_ERR_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

void lsx_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns);
}

void lsx_set_deterministic(int on) { g_deterministic.store(on != 0 ? 1 : 0); }

int lsx_sync_status(lsx_stream_t stream) {
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return LSX_ERR_LAUNCH;
  int word = 0;
  if (cudaMemcpy(&word, ctx.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LSX_ERR_LAUNCH;
  const int zero = 0;
  if (cudaMemcpy(ctx.status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return LSX_ERR_LAUNCH;
  return word;
}

// ------------------------------------------------------------ attn_merge
int attn_merge(const lsx_tensor* o_a, const lsx_tensor* lse_a,
               const lsx_tensor* o_b, const lsx_tensor* lse_b,
               const lsx_tensor* o_out, const lsx_tensor* lse_out,
               lsx_stream_t stream) {
  LSX_TRY(check_view(o_a));
  LSX_TRY(check_view(o_b));
  LSX_TRY(check_view(o_out));
  if (!same_bhn_d(o_a, o_b) || !same_bhn_d(o_a, o_out)) return LSX_ERR_SHAPE;
  if (o_a->D != 64 && o_a->D != 128) return LSX_ERR_UNSUPPORTED;
  LSX_TRY(check_row_aligned(o_a));
  LSX_TRY(check_row_aligned(o_b));
  LSX_TRY(check_row_aligned(o_out));
  LSX_TRY(check_lse(lse_a, o_a));
  LSX_TRY(check_lse(lse_b, o_a));
  LSX_TRY(check_lse(lse_out, o_a));
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  return launch_merge(*o_a, *lse_a, *o_b, *lse_b, *o_out, *lse_out, ctx,
                      as_stream(stream));
}

// ------------------------------------------------------- attn_tree_merge
int attn_tree_merge(const lsx_tensor* o_parts, int64_t part_stride_o,
                    const lsx_tensor* lse_parts, int64_t part_stride_lse,
                    int n_parts, const lsx_tensor* o_out,
                    const lsx_tensor* lse_out, lsx_stream_t stream) {
  LSX_TRY(check_view(o_parts));
  LSX_TRY(check_view(o_out));
  if (!same_bhn_d(o_parts, o_out)) return LSX_ERR_SHAPE;
  if (o_parts->D != 64 && o_parts->D != 128) return LSX_ERR_UNSUPPORTED;
  if (n_parts < 1 || n_parts > 4096) return LSX_ERR_UNSUPPORTED;
  if (part_stride_o < 0 || part_stride_lse < 0) return LSX_ERR_SHAPE;
  LSX_TRY(check_row_aligned(o_parts));
  LSX_TRY(check_row_aligned(o_out));
  if (part_stride_o % (16 / elem_size(o_parts->dtype)) != 0) return LSX_ERR_ALIGN;
  LSX_TRY(check_lse(lse_parts, o_parts));
  lsx_tensor lo_none{};
  const lsx_tensor* lo = lse_out;
  if (lse_out == nullptr || lse_out->data == nullptr) {
    lo_none = *o_out;
    lo_none.data = nullptr;
    lo_none.D = 1;
    lo = &lo_none;
  } else {
    LSX_TRY(check_lse(lse_out, o_parts));
  }
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  return launch_tree_merge(*o_parts, part_stride_o, *lse_parts, part_stride_lse,
                           n_parts, *o_out, *lo, ctx, as_stream(stream));
}

// -------------------------------------------------------- attn_chunk_fwd
size_t attn_chunk_fwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k) {
  if (q == nullptr || k == nullptr || q->dtype != LSX_BF16) return 0;
  return fwd_tc_workspace_bytes(*k) + 256;
}

int attn_chunk_fwd(const lsx_tensor* q, const lsx_tensor* k,
                   const lsx_tensor* v, int64_t q_off, int64_t kv_off,
                   int causal, float scale, const lsx_tensor* o,
                   const lsx_tensor* lse, int accumulate, void* workspace,
                   size_t workspace_bytes, lsx_stream_t stream) {
  LSX_TRY(check_qkv(q, k, v));
  LSX_TRY(check_view(o));
  if (o->B != q->B || o->H != q->H || o->N != q->N || o->D != q->D) return LSX_ERR_SHAPE;
  if (q->dtype == LSX_F32 && o->dtype != LSX_F32) return LSX_ERR_DTYPE;
  LSX_TRY(check_row_aligned(o));
  LSX_TRY(check_lse(lse, q));
  if (q_off < 0 || kv_off < 0) return LSX_ERR_SHAPE;
  // optional workspace: NULL, or large enough for the transposed copy of V
  void* vt = nullptr;
  if (workspace != nullptr && q->dtype == LSX_BF16) {
    if (workspace_bytes < attn_chunk_fwd_workspace_size(q, k)) return LSX_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return LSX_ERR_ALIGN;
    vt = workspace;
  }
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  const float sc = resolve_scale(scale, q->D);
  cudaStream_t s = as_stream(stream);
  if (q->N == 0) return LSX_OK;
  if (k->N == 0) return accumulate ? LSX_OK : launch_fill_empty(*o, *lse, ctx, s);
  if (q->dtype == LSX_F32)
    return launch_simt_fwd(*q, *k, *v, q_off, kv_off, causal != 0, sc, *o, *lse,
                           accumulate != 0, ctx, s);
  return launch_fwd_tc(*q, *k, *v, q_off, kv_off, causal != 0, sc, *o, *lse,
                       accumulate != 0, vt, ctx, s);
}

// -------------------------------------------------------- attn_chunk_bwd
size_t attn_chunk_bwd_min_workspace_size(const lsx_tensor* q, const lsx_tensor* k) {
  (void)k;
  if (q == nullptr) return 0;
  const int64_t rows = q->B * q->H * q->N;
  return (static_cast<size_t>(rows > 0 ? rows : 0) * sizeof(float) + 255) / 256 * 256;
}

size_t attn_chunk_bwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k) {
  if (q == nullptr || k == nullptr) return 0;
  size_t n = attn_chunk_bwd_min_workspace_size(q, k);
  if (q->dtype == LSX_BF16) n += bwd_tc_copies_bytes(*q, *k);
  return n;
}

// attn_chunk_bwd, and attn_chunked_bwd's split form (split != NULL: the
// full workspace's copies are required and its partials follow them)
static int chunk_bwd_impl(const lsx_tensor* q, const lsx_tensor* k,
                          const lsx_tensor* v, const lsx_tensor* o,
                          const lsx_tensor* lse, const lsx_tensor* d_o,
                          int64_t q_off, int64_t kv_off, int causal, float scale,
                          const lsx_tensor* dq, const lsx_tensor* dk,
                          const lsx_tensor* dv, int accumulate, void* workspace,
                          size_t workspace_bytes, lsx_stream_t stream, const BwdSplit* split) {
  LSX_TRY(check_qkv(q, k, v));
  LSX_TRY(check_view(o));
  LSX_TRY(check_view(d_o));
  LSX_TRY(check_view(dq));
  LSX_TRY(check_view(dk));
  LSX_TRY(check_view(dv));
  if (!same_bhn_d(o, q) || !same_bhn_d(d_o, q) || !same_bhn_d(dq, q) ||
      !same_bhn_d(dk, k) || !same_bhn_d(dv, k))
    return LSX_ERR_SHAPE;
  if (d_o->dtype != q->dtype) return LSX_ERR_DTYPE;
  if (q->dtype == LSX_F32 &&
      (dq->dtype != LSX_F32 || dk->dtype != LSX_F32 || dv->dtype != LSX_F32 ||
       o->dtype != LSX_F32))
    return LSX_ERR_DTYPE;
  LSX_TRY(check_row_aligned(o));
  LSX_TRY(check_row_aligned(d_o));
  LSX_TRY(check_row_aligned(dq));
  LSX_TRY(check_row_aligned(dk));
  LSX_TRY(check_row_aligned(dv));
  LSX_TRY(check_lse(lse, q));
  if (q_off < 0 || kv_off < 0) return LSX_ERR_SHAPE;
  const size_t need = attn_chunk_bwd_min_workspace_size(q, k);
  if (workspace == nullptr || workspace_bytes < need) return LSX_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return LSX_ERR_ALIGN;
  // room for the sequence-contiguous copies: the faster operand layout
  BwdCopies copies;
  if (q->dtype == LSX_BF16 && workspace_bytes >= attn_chunk_bwd_workspace_size(q, k))
    copies = bwd_tc_copies(*q, *k, static_cast<char*>(workspace) + need);
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  const float sc = resolve_scale(scale, q->D);
  cudaStream_t s = as_stream(stream);
  if (q->N == 0 || k->N == 0) {
    if (accumulate) return LSX_OK;
    if (q->N > 0) LSX_TRY(launch_zero(*dq, ctx, s));
    if (k->N > 0) {
      LSX_TRY(launch_zero(*dk, ctx, s));
      LSX_TRY(launch_zero(*dv, ctx, s));
    }
    return LSX_OK;
  }
  float* delta = static_cast<float*>(workspace);
  LSX_TRY(launch_row_dot(*o, *d_o, delta, copies.stats, lse, sc, ctx, s));
  if (q->dtype == LSX_F32)
    return launch_simt_bwd(*q, *k, *v, *lse, *d_o, delta, q_off, kv_off,
                           causal != 0, sc, *dq, *dk, *dv, accumulate != 0, ctx, s);
  if (split != nullptr) {
    if (copies.stats.rows == nullptr || accumulate) return LSX_ERR_WORKSPACE;
    return launch_bwd_tc_split(*q, *k, *v, *lse, *d_o, delta, copies, q_off, kv_off,
                               causal != 0, sc, *dq, *dk, *dv, *split, ctx, s);
  }
  return launch_bwd_tc(*q, *k, *v, *lse, *d_o, delta, copies, q_off, kv_off,
                       causal != 0, sc, *dq, *dk, *dv, accumulate != 0, ctx, s);
}

int attn_chunk_bwd(const lsx_tensor* q, const lsx_tensor* k,
                   const lsx_tensor* v, const lsx_tensor* o,
                   const lsx_tensor* lse, const lsx_tensor* d_o,
                   int64_t q_off, int64_t kv_off, int causal, float scale,
                   const lsx_tensor* dq, const lsx_tensor* dk,
                   const lsx_tensor* dv, int accumulate, void* workspace,
                   size_t workspace_bytes, lsx_stream_t stream) {
  return chunk_bwd_impl(q, k, v, o, lse, d_o, q_off, kv_off, causal, scale, dq, dk, dv,
                        accumulate, workspace, workspace_bytes, stream, nullptr);
}

// ------------------------------------------- whole-sequence chunked calls
// Rows split into key pieces (Lean Attention abstract: the partials of one
// row, computed by different workers, combine exactly by the associative
// merge).  The persistent forward deals its query pairs over the SMs
// longest first; with fewer pairs than SMs (few heads, long rows) some SMs
// have nothing to do and the longest rows set the launch's time.  The pairs'
// visible key tiles are then cut into pieces of piece_w tiles, sized for
// about four pieces of work per SM and at most 32 pieces per row (one warp
// merges them), and the merge kernel combines each row's pieces.  (Measured:
// one 32K head, 128 pairs, 0.50 -> 0.36 ms; with 256 pairs the unsplit deal
// was already balanced and splitting lost.)
static bool plan_split(const lsx_tensor& q, const lsx_tensor& k, int causal, int sm_count,
                       FwdSplit* out) {
  if (q.dtype != LSX_BF16 || q.N <= 0 || k.N <= 0 || sm_count <= 0) return false;
  if (q.D != 64 && q.D != 128) return false;
  const int64_t n_pairs = ceil_div(q.N, 256);
  if (q.B * q.H * n_pairs >= static_cast<int64_t>(sm_count)) return false;
  int64_t total = 0, longest = 0;
  for (int64_t pr = 0; pr < n_pairs; ++pr) {
    const int64_t a = fwd_kv_tiles(2 * pr, q.N, k.N, 0, 0, causal);
    const int64_t b = fwd_kv_tiles(2 * pr + 1, q.N, k.N, 0, 0, causal);
    const int64_t m = a > b ? a : b;
    total += m;
    if (m > longest) longest = m;
  }
  total *= q.B * q.H;
  int64_t w = ceil_div(total, 4 * static_cast<int64_t>(sm_count));
  if (w < 4) w = 4;
  if (ceil_div(longest, w) > 32) w = ceil_div(longest, 32);
  const int64_t kmax = ceil_div(longest, w);
  if (kmax < 2) return false;
  out->piece_w = w;
  out->kmax = kmax;
  return true;
}

// bytes of the partials of a split (O, then LSE), each region 256-aligned
static size_t split_bytes(const lsx_tensor& q, const FwdSplit& sp, size_t* o_bytes) {
  const size_t rows = static_cast<size_t>(sp.kmax) * q.B * q.H * q.N;
  *o_bytes = (rows * q.D * sizeof(float) + 255) / 256 * 256;
  return *o_bytes + (rows * sizeof(float) + 255) / 256 * 256;
}

static int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t attn_chunked_fwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k,
                                       int64_t chunk_len, int causal) {
  (void)chunk_len;
  const size_t base = attn_chunk_fwd_workspace_size(q, k);
  if (base == 0) return 0;
  FwdSplit sp;
  if (!plan_split(*q, *k, causal, current_sm_count(), &sp)) return base;
  size_t o_bytes;
  return base + split_bytes(*q, sp, &o_bytes);
}

int attn_chunked_fwd(const lsx_tensor* q, const lsx_tensor* k,
                     const lsx_tensor* v, int64_t chunk_len, int causal,
                     float scale, const lsx_tensor* o, const lsx_tensor* lse,
                     void* workspace, size_t workspace_bytes,
                     lsx_stream_t stream) {
  LSX_TRY(check_qkv(q, k, v));
  if (q->N != k->N) return LSX_ERR_SHAPE;
  if (chunk_len <= 0 || chunk_len % 128 != 0) return LSX_ERR_UNSUPPORTED;
  // Split the rows when the workspace holds their partials (see plan_split);
  // otherwise one persistent launch covers every visible chunk pair (see
  // fwd_tc.cu): the chunk length sets no boundary the online softmax could
  // not cross.
  FwdSplit sp;
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  const size_t base = attn_chunk_fwd_workspace_size(q, k);
  size_t o_bytes = 0;
  if (workspace != nullptr && base > 0 && plan_split(*q, *k, causal, ctx.sm_count, &sp) &&
      workspace_bytes >= base + split_bytes(*q, sp, &o_bytes)) {
    LSX_TRY(check_view(o));
    if (o->B != q->B || o->H != q->H || o->N != q->N || o->D != q->D) return LSX_ERR_SHAPE;
    LSX_TRY(check_row_aligned(o));
    LSX_TRY(check_lse(lse, q));
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return LSX_ERR_ALIGN;
    char* ws = static_cast<char*>(workspace);
    sp.part_o = reinterpret_cast<float*>(ws + base);
    sp.part_lse = reinterpret_cast<float*>(ws + base + o_bytes);
    const float sc = resolve_scale(scale, q->D);
    cudaStream_t s = as_stream(stream);
    LSX_TRY(launch_fwd_tc_split(*q, *k, *v, 0, 0, causal != 0, sc, *o, *lse, workspace, sp,
                                ctx, s));
    return launch_merge_pieces(sp, 0, 0, causal != 0, k->N, *o, *lse, ctx, s);
  }
  return attn_chunk_fwd(q, k, v, 0, 0, causal, scale, o, lse, 0, workspace,
                        workspace_bytes, stream);
}

// The backward's counterpart of plan_split: its items are (b, kv head, key
// tile), each walking the query tiles that see the key tile for every head
// of the group.  With fewer items than SMs those steps are cut into pieces
// (about four pieces of work per SM, at most 32 per item); each piece
// writes partial dK, dV that a sum kernel adds up.  Not in deterministic
// mode (the partial sums would be one more reduction order to pin).
static bool plan_split_bwd(const lsx_tensor& q, const lsx_tensor& k, int causal,
                           const DeviceCtx& ctx, BwdSplit* out) {
  if (ctx.deterministic || ctx.sm_count <= 0) return false;
  if (q.dtype != LSX_BF16 || q.N <= 0 || k.N <= 0 || (q.D != 64 && q.D != 128)) return false;
  const int64_t n_kt = ceil_div(k.N, 128), n_qt = ceil_div(q.N, 128);
  if (k.B * k.H * n_kt >= static_cast<int64_t>(ctx.sm_count)) return false;
  const int64_t group = q.H / k.H;
  int64_t total = 0, longest = 0;
  for (int64_t j = 0; j < n_kt; ++j) {
    // query tiles that see key tile j (offsets 0, as in the chunked call)
    int64_t i0 = 0;
    if (causal) {
      const int64_t need = 128 * j;
      i0 = need > q.N - 1 ? n_qt : need / 128;
    }
    const int64_t steps = (n_qt - i0) * group;
    total += steps;
    if (steps > longest) longest = steps;
  }
  total *= k.B * k.H;
  int64_t w = ceil_div(total, 4 * static_cast<int64_t>(ctx.sm_count));
  if (w < 4) w = 4;
  if (ceil_div(longest, w) > 32) w = ceil_div(longest, 32);
  const int64_t kmax = ceil_div(longest, w);
  if (kmax < 2) return false;
  out->piece_w = w;
  out->kmax = kmax;
  return true;
}

static size_t split_bwd_bytes(const lsx_tensor& k, const BwdSplit& sp, size_t* one) {
  *one = (static_cast<size_t>(sp.kmax) * k.B * k.H * k.N * k.D * sizeof(float) + 255) / 256 * 256;
  return 2 * *one;
}

size_t attn_chunked_bwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k,
                                       int64_t chunk_len, int causal) {
  (void)chunk_len;
  const size_t base = attn_chunk_bwd_workspace_size(q, k);
  if (base == 0 || q == nullptr || k == nullptr || q->dtype != LSX_BF16) return base;
  DeviceCtx ctx;
  if (device_ctx(&ctx) != LSX_OK) return base;
  BwdSplit sp;
  if (!plan_split_bwd(*q, *k, causal, ctx, &sp)) return base;
  size_t one;
  return base + split_bwd_bytes(*k, sp, &one);
}

int attn_chunked_bwd(const lsx_tensor* q, const lsx_tensor* k,
                     const lsx_tensor* v, const lsx_tensor* o,
                     const lsx_tensor* lse, const lsx_tensor* d_o,
                     int64_t chunk_len, int causal, float scale,
                     const lsx_tensor* dq, const lsx_tensor* dk,
                     const lsx_tensor* dv, void* workspace,
                     size_t workspace_bytes, lsx_stream_t stream) {
  LSX_TRY(check_qkv(q, k, v));
  if (q->N != k->N) return LSX_ERR_SHAPE;
  if (chunk_len <= 0 || chunk_len % 128 != 0) return LSX_ERR_UNSUPPORTED;
  // key columns split into pieces when the workspace holds their partials
  // (see plan_split_bwd); otherwise one persistent launch
  BwdSplit sp;
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  const size_t base = attn_chunk_bwd_workspace_size(q, k);
  size_t one = 0;
  if (workspace != nullptr && q->dtype == LSX_BF16 && plan_split_bwd(*q, *k, causal, ctx, &sp) &&
      workspace_bytes >= base + split_bwd_bytes(*k, sp, &one)) {
    char* ws = static_cast<char*>(workspace);
    sp.part_dk = reinterpret_cast<float*>(ws + base);
    sp.part_dv = reinterpret_cast<float*>(ws + base + one);
    return chunk_bwd_impl(q, k, v, o, lse, d_o, 0, 0, causal, scale, dq, dk, dv, 0, workspace,
                          base, stream, &sp);
  }
  return attn_chunk_bwd(q, k, v, o, lse, d_o, 0, 0, causal, scale, dq, dk, dv, 0,
                        workspace, workspace_bytes, stream);
}

// ------------------------------------------------- block-sparse attention
// Workspace: [V^T copy (forward) | delta, K^T copy, row statistics
// (backward)] then the block lists, each part 256-byte aligned.
size_t attn_block_sparse_fwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k) {
  if (q == nullptr || k == nullptr || q->dtype != LSX_BF16) return 0;
  return attn_chunk_fwd_workspace_size(q, k) + block_lists_bytes(q->N, k->N);
}

size_t attn_block_sparse_bwd_workspace_size(const lsx_tensor* q, const lsx_tensor* k) {
  if (q == nullptr || k == nullptr || q->dtype != LSX_BF16) return 0;
  return attn_chunk_bwd_workspace_size(q, k) + block_lists_bytes(q->N, k->N);
}

int attn_block_sparse_fwd(const lsx_tensor* q, const lsx_tensor* k, const lsx_tensor* v,
                          const uint8_t* block_mask, int causal, float scale,
                          const lsx_tensor* o, const lsx_tensor* lse, void* workspace,
                          size_t workspace_bytes, lsx_stream_t stream) {
  LSX_TRY(check_qkv(q, k, v));
  if (q->dtype != LSX_BF16) return LSX_ERR_DTYPE;
  if (block_mask == nullptr) return LSX_ERR_NULL;
  LSX_TRY(check_view(o));
  if (o->B != q->B || o->H != q->H || o->N != q->N || o->D != q->D) return LSX_ERR_SHAPE;
  LSX_TRY(check_row_aligned(o));
  LSX_TRY(check_lse(lse, q));
  if (workspace == nullptr || workspace_bytes < attn_block_sparse_fwd_workspace_size(q, k))
    return LSX_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return LSX_ERR_ALIGN;
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  const float sc = resolve_scale(scale, q->D);
  cudaStream_t s = as_stream(stream);
  if (q->N == 0) return LSX_OK;
  if (k->N == 0) return launch_fill_empty(*o, *lse, ctx, s);
  void* vt = workspace;
  void* lists = static_cast<char*>(workspace) + attn_chunk_fwd_workspace_size(q, k);
  BlockLists bl;
  LSX_TRY(build_block_lists(block_mask, q->N, k->N, causal != 0, lists, &bl, ctx, s));
  return launch_fwd_tc(*q, *k, *v, 0, 0, causal != 0, sc, *o, *lse, 0, vt, ctx, s, &bl);
}

int attn_block_sparse_bwd(const lsx_tensor* q, const lsx_tensor* k, const lsx_tensor* v,
                          const lsx_tensor* o, const lsx_tensor* lse, const lsx_tensor* d_o,
                          const uint8_t* block_mask, int causal, float scale,
                          const lsx_tensor* dq, const lsx_tensor* dk, const lsx_tensor* dv,
                          void* workspace, size_t workspace_bytes, lsx_stream_t stream) {
  LSX_TRY(check_qkv(q, k, v));
  if (q->dtype != LSX_BF16) return LSX_ERR_DTYPE;
  if (block_mask == nullptr) return LSX_ERR_NULL;
  LSX_TRY(check_view(o));
  LSX_TRY(check_view(d_o));
  LSX_TRY(check_view(dq));
  LSX_TRY(check_view(dk));
  LSX_TRY(check_view(dv));
  if (!same_bhn_d(o, q) || !same_bhn_d(d_o, q) || !same_bhn_d(dq, q) ||
      !same_bhn_d(dk, k) || !same_bhn_d(dv, k))
    return LSX_ERR_SHAPE;
  if (d_o->dtype != q->dtype) return LSX_ERR_DTYPE;
  LSX_TRY(check_row_aligned(o));
  LSX_TRY(check_row_aligned(d_o));
  LSX_TRY(check_row_aligned(dq));
  LSX_TRY(check_row_aligned(dk));
  LSX_TRY(check_row_aligned(dv));
  LSX_TRY(check_lse(lse, q));
  if (workspace == nullptr || workspace_bytes < attn_block_sparse_bwd_workspace_size(q, k))
    return LSX_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return LSX_ERR_ALIGN;
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  const float sc = resolve_scale(scale, q->D);
  cudaStream_t s = as_stream(stream);
  if (q->N == 0 || k->N == 0) {
    if (q->N > 0) LSX_TRY(launch_zero(*dq, ctx, s));
    if (k->N > 0) {
      LSX_TRY(launch_zero(*dk, ctx, s));
      LSX_TRY(launch_zero(*dv, ctx, s));
    }
    return LSX_OK;
  }
  const size_t need = attn_chunk_bwd_min_workspace_size(q, k);
  const BwdCopies copies = bwd_tc_copies(*q, *k, static_cast<char*>(workspace) + need);
  void* lists = static_cast<char*>(workspace) + attn_chunk_bwd_workspace_size(q, k);
  BlockLists bl;
  LSX_TRY(build_block_lists(block_mask, q->N, k->N, causal != 0, lists, &bl, ctx, s));
  float* delta = static_cast<float*>(workspace);
  LSX_TRY(launch_row_dot(*o, *d_o, delta, copies.stats, lse, sc, ctx, s));
  return launch_bwd_tc(*q, *k, *v, *lse, *d_o, delta, copies, 0, 0, causal != 0, sc, *dq,
                       *dk, *dv, 0, ctx, s, &bl);
}

// ----------------------------------------------------------- attn_decode
size_t attn_decode_workspace_size(const lsx_tensor* q, const lsx_tensor* kc,
                                  int64_t chunk_len) {
  if (q == nullptr || kc == nullptr || chunk_len <= 0) return 0;
  const int64_t parts = ceil_div(kc->N, chunk_len);
  const int64_t rows = q->B * q->H;
  // partial O [parts][rows][D] f32, then partial LSE [parts][rows] f32
  const size_t o_bytes = static_cast<size_t>(parts * rows * q->D) * sizeof(float);
  const size_t l_bytes = static_cast<size_t>(parts * rows) * sizeof(float);
  return ((o_bytes + 255) / 256) * 256 + ((l_bytes + 255) / 256) * 256;
}

int attn_decode(const lsx_tensor* q, const lsx_tensor* kc,
                const lsx_tensor* vc, int64_t chunk_len, float scale,
                const lsx_tensor* o, const lsx_tensor* lse, void* workspace,
                size_t workspace_bytes, lsx_stream_t stream) {
  LSX_TRY(check_qkv(q, kc, vc));
  if (q->dtype != LSX_BF16) return LSX_ERR_DTYPE;
  if (q->N != 1 || q->D != 128) return LSX_ERR_UNSUPPORTED;
  {
    const int64_t g = q->H / kc->H;
    if (g != 1 && g != 2 && g != 4 && g != 8) return LSX_ERR_UNSUPPORTED;
  }
  LSX_TRY(check_view(o));
  if (!same_bhn_d(o, q)) return LSX_ERR_SHAPE;
  LSX_TRY(check_row_aligned(o));
  LSX_TRY(check_lse(lse, q));
  if (chunk_len <= 0 || chunk_len % 128 != 0) return LSX_ERR_UNSUPPORTED;
  const int64_t parts = ceil_div(kc->N, chunk_len);
  if (parts > 4096) return LSX_ERR_UNSUPPORTED;
  const size_t need = attn_decode_workspace_size(q, kc, chunk_len);
  if (workspace == nullptr || workspace_bytes < need) return LSX_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return LSX_ERR_ALIGN;
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  cudaStream_t s = as_stream(stream);
  if (kc->N == 0) return launch_fill_empty(*o, *lse, ctx, s);
  const float sc = resolve_scale(scale, q->D);
  const int64_t rows = q->B * q->H;
  float* part_o = static_cast<float*>(workspace);
  const size_t o_bytes = static_cast<size_t>(parts * rows * q->D) * sizeof(float);
  float* part_l = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           ((o_bytes + 255) / 256) * 256);
  LSX_TRY(launch_decode_partials(*q, *kc, *vc, chunk_len, sc, part_o, part_l, ctx, s));
  // partial p of query row (b, h) sits at part_o[(p * rows + b*H + h) * D]
  lsx_tensor po{part_o, LSX_F32, 0, q->B, q->H, 1, q->D, q->H * q->D, q->D, q->D};
  lsx_tensor pl{part_l, LSX_F32, 0, q->B, q->H, 1, 1, q->H, 1, 1};
  return launch_tree_merge(po, rows * q->D, pl, rows, static_cast<int>(parts), *o,
                           *lse, ctx, s);
}

// ------------------------------------------------------- attn_decode_tree
namespace {
int64_t tree_parts(const lsx_tensor* pk, const lsx_tensor* sk, int64_t chunk_len) {
  const int64_t ns = (sk == nullptr || sk->data == nullptr) ? 0 : sk->N;
  return ceil_div(pk->N, chunk_len) + ceil_div(ns, chunk_len);
}
}  // namespace

size_t attn_decode_tree_workspace_size(const lsx_tensor* q, const lsx_tensor* pk,
                                       const lsx_tensor* sk, int64_t chunk_len) {
  if (q == nullptr || pk == nullptr || chunk_len <= 0) return 0;
  const int64_t parts = tree_parts(pk, sk, chunk_len);
  const int64_t rows = q->B * q->H;
  const size_t o_bytes = static_cast<size_t>(parts * rows * q->D) * sizeof(float);
  const size_t l_bytes = static_cast<size_t>(parts * rows) * sizeof(float);
  return ((o_bytes + 255) / 256) * 256 + ((l_bytes + 255) / 256) * 256;
}

int attn_decode_tree(const lsx_tensor* q, const lsx_tensor* pk, const lsx_tensor* pv,
                     const lsx_tensor* sk, const lsx_tensor* sv, int64_t chunk_len,
                     float scale, const lsx_tensor* o, const lsx_tensor* lse, void* workspace,
                     size_t workspace_bytes, lsx_stream_t stream) {
  if (q == nullptr || pk == nullptr) return LSX_ERR_NULL;
  if (pk->B != 1) return LSX_ERR_SHAPE;
  {
    lsx_tensor q1 = *q;  // the prefix is one cache for every branch
    q1.B = 1;
    LSX_TRY(check_qkv(&q1, pk, pv));
    LSX_TRY(check_view(q));
  }
  if (q->dtype != LSX_BF16) return LSX_ERR_DTYPE;
  if (q->N != 1 || q->D != 128) return LSX_ERR_SHAPE;
  const bool has_suffix = sk != nullptr && sk->data != nullptr && sk->N > 0;
  if (has_suffix) {
    LSX_TRY(check_qkv(q, sk, sv));
    if (sk->B != q->B || sk->H != pk->H) return LSX_ERR_SHAPE;
  }
  {
    const int64_t g = q->H / pk->H;
    if (g != 1 && g != 2 && g != 4 && g != 8) return LSX_ERR_UNSUPPORTED;
  }
  LSX_TRY(check_view(o));
  if (!same_bhn_d(o, q)) return LSX_ERR_SHAPE;
  LSX_TRY(check_row_aligned(o));
  LSX_TRY(check_lse(lse, q));
  if (chunk_len <= 0 || chunk_len % 128 != 0) return LSX_ERR_UNSUPPORTED;
  const int64_t parts = tree_parts(pk, has_suffix ? sk : nullptr, chunk_len);
  if (parts > 4096) return LSX_ERR_UNSUPPORTED;
  const size_t need = attn_decode_tree_workspace_size(q, pk, has_suffix ? sk : nullptr, chunk_len);
  if (workspace == nullptr || workspace_bytes < need) return LSX_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return LSX_ERR_ALIGN;
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  cudaStream_t s = as_stream(stream);
  if (parts == 0) return launch_fill_empty(*o, *lse, ctx, s);
  const float sc = resolve_scale(scale, q->D);
  const int64_t rows = q->B * q->H;
  float* part_o = static_cast<float*>(workspace);
  const size_t o_bytes = static_cast<size_t>(parts * rows * q->D) * sizeof(float);
  float* part_l = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           ((o_bytes + 255) / 256) * 256);
  const int64_t p_parts = ceil_div(pk->N, chunk_len);
  if (p_parts > 0)
    LSX_TRY(launch_decode_shared(*q, *pk, *pv, chunk_len, sc, part_o, part_l, ctx, s, 0));
  if (has_suffix)
    LSX_TRY(launch_decode_partials(*q, *sk, *sv, chunk_len, sc, part_o, part_l, ctx, s,
                                   p_parts));
  lsx_tensor po{part_o, LSX_F32, 0, q->B, q->H, 1, q->D, q->H * q->D, q->D, q->D};
  lsx_tensor pl{part_l, LSX_F32, 0, q->B, q->H, 1, 1, q->H, 1, 1};
  return launch_tree_merge(po, rows * q->D, pl, rows, static_cast<int>(parts), *o, *lse, ctx,
                           s);
}

// ----------------------------------------------------------------- timing
int lsx_timing_enable(int on) {
  g_timing.store(on != 0);
  return LSX_OK;
}

int lsx_timing_reset(void) {
  std::lock_guard<std::mutex> lk(g_tmu);
  for (auto& t : g_launches) {
    g_event_pool.push_back(t.a);
    g_event_pool.push_back(t.b);
  }
  g_launches.clear();
  return LSX_OK;
}

int lsx_timing_report(char* buf, size_t n) {
  if (buf == nullptr || n == 0) return LSX_ERR_NULL;
  std::lock_guard<std::mutex> lk(g_tmu);
  double total[kKidCount] = {0};
  int64_t count[kKidCount] = {0};
  for (auto& t : g_launches) {
    if (cudaEventSynchronize(t.b) != cudaSuccess) return LSX_ERR_LAUNCH;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.a, t.b) != cudaSuccess) return LSX_ERR_LAUNCH;
    total[t.kid] += ms;
    count[t.kid] += 1;
  }
  size_t used = 0;
  int reported = 0;
  buf[0] = '\0';
  for (int k = 0; k < kKidCount; ++k) {
    if (count[k] == 0) continue;
    const int w = snprintf(buf + used, n - used, "%s %lld %.6f\n", kKernelNames[k],
                           static_cast<long long>(count[k]), total[k]);
    if (w < 0 || static_cast<size_t>(w) >= n - used) break;
    used += static_cast<size_t>(w);
    ++reported;
  }
  return reported;
}

// --------------------------------------------------------- schedule trace
int lsx_trace_enable(void* buf, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_trmu);
  if (buf != nullptr && reinterpret_cast<uintptr_t>(buf) % 8 != 0) return LSX_ERR_ALIGN;
  g_trace_buf = static_cast<uint64_t*>(buf);
  g_trace_cap = buf == nullptr ? 0 : bytes / sizeof(uint64_t);
  g_trace_used = 0;
  return LSX_OK;
}

size_t lsx_trace_used(void) {
  std::lock_guard<std::mutex> lk(g_trmu);
  return g_trace_used * sizeof(uint64_t);
}

// ------------------------------------------------------------ diagnostics
int lsx_schedule_stats(int64_t B, int64_t H, int64_t N, int64_t chunk_len,
                       int causal, int n_workers, int64_t* out) {
  if (out == nullptr) return LSX_ERR_NULL;
  if (B <= 0 || H <= 0 || N <= 0 || n_workers <= 0) return LSX_ERR_SHAPE;
  if (chunk_len <= 0 || chunk_len % 128 != 0) return LSX_ERR_UNSUPPORTED;
  const int64_t n_qpairs = ceil_div(N, 256);
  const int64_t n_items = n_qpairs * B * H;
  const int64_t G = n_items < n_workers ? n_items : n_workers;
  std::vector<int64_t> load(static_cast<size_t>(G), 0);
  int64_t total = 0;
  for (int64_t c = 0; c < G; ++c) {
    for (int64_t r = 0;; ++r) {
      const int64_t it = snake_item(c, r, G);
      if (it >= n_items) break;
      int64_t rank, bh;
      banded_item(it, n_qpairs, B * H, &rank, &bh);
      const int64_t pair = n_qpairs - 1 - rank;
      const int64_t a = fwd_kv_tiles(2 * pair, N, N, 0, 0, causal);
      const int64_t b = fwd_kv_tiles(2 * pair + 1, N, N, 0, 0, causal);
      const int64_t cost = a + b;  // one S and one P.V product per tile row
      load[static_cast<size_t>(c)] += cost;
      total += cost;
    }
  }
  out[0] = *std::max_element(load.begin(), load.end());
  out[1] = ceil_div(total, n_workers);
  out[2] = total;
  return LSX_OK;
}

}  // extern "C"

// ------------------------------------------------ bounded-wait self-test
namespace lsx {
namespace {
__global__ void bounded_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);  // nobody ever arrives
    fence_barrier_init();
  }
  __syncthreads();
  const WaitGuard g{status, limit_ns, &abort_flag};
  (void)mbar_wait(&bar, 0, g);
  __syncthreads();
}
}  // namespace
}  // namespace lsx

extern "C" int lsx_selftest_bounded_wait(lsx_stream_t stream) {
  DeviceCtx ctx;
  LSX_TRY(device_ctx(&ctx));
  bounded_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(ctx.status, ctx.wait_ns);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}
