// internal.h -- declarations shared by the translation units of liblsx.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lsx.h"

namespace lsx {

// Per-device facts the launchers need.
struct DeviceCtx {
  int device;
  int sm_count;
  int* status;        // device address of this device's status word
  uint64_t wait_ns;   // bound of every device-side wait
  int deterministic;  // backward: owner-computes dQ (no fp32 reductions)
};

// Fills ctx for the current device; returns LSX_OK or LSX_ERR_DEVICE.
int device_ctx(DeviceCtx* ctx);

// Optional per-kernel timing (lsx_timing_enable): a CUDA event pair is
// recorded on the launching stream around every launch of kernel `kid`.
enum KernelId {
  kKidFwdTc = 0, kKidDkdv, kKidDq, kKidRowDot, kKidMerge, kKidTreeMerge,
  kKidDecode, kKidSimtFwd, kKidSimtBwd, kKidFill, kKidTranspose, kKidBlockLists,
  kKidBwdFused, kKidDqConvert, kKidCount
};

// Sequence-contiguous copies (layout.cu): a bf16 [B, H, N, D] view is
// written densely as [B, H, D, Np], Np = N rounded up to a multiple of 8.
int64_t transposed_row_len(int64_t n);
size_t transposed_bytes(const lsx_tensor& t);
int launch_transpose(const lsx_tensor& in, void* out, cudaStream_t s);
void timing_begin(int kid, cudaStream_t s);
void timing_end(int kid, cudaStream_t s);

// Optional per-CTA trace of the persistent kernels (lsx_trace_enable).  A
// launch of kernel `kid` on `grid` CTAs asks for a record; NULL means no
// tracing (disabled, or the caller's buffer is full).  The kernel writes the
// record itself: words [0..2] = kid, grid, work items; then for CTA c the
// words [3 + 3c .. 5 + 3c] = %globaltimer when it starts its first item,
// %globaltimer when it has finished its last, and the items it ran.
uint64_t* trace_record(int kid, int64_t grid);
constexpr int64_t trace_words(int64_t grid) { return 3 + 3 * grid; }

// Record writes, by thread 0 of each CTA: trace_begin after the set-up,
// trace_items when its loader has gone through its items, trace_end once
// every role has left its loop.
__device__ __forceinline__ uint64_t* trace_cta(uint64_t* rec) {
  return rec + 3 + 3 * static_cast<int64_t>(blockIdx.x);
}
__device__ __forceinline__ void trace_begin(uint64_t* rec, int kid, int64_t n_items,
                                            uint64_t now) {
  if (blockIdx.x == 0) {
    rec[0] = static_cast<uint64_t>(kid);
    rec[1] = gridDim.x;
    rec[2] = static_cast<uint64_t>(n_items);
  }
  trace_cta(rec)[0] = now;
}
__device__ __forceinline__ void trace_items(uint64_t* rec, int64_t done) {
  trace_cta(rec)[2] = static_cast<uint64_t>(done);
}
__device__ __forceinline__ void trace_end(uint64_t* rec, uint64_t now) {
  trace_cta(rec)[1] = now;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Element offset of (b, h, n, 0) in a view.
__host__ __device__ inline int64_t view_off(const lsx_tensor& t, int64_t b,
                                            int64_t h, int64_t n) {
  return b * t.stride_b + h * t.stride_h + n * t.stride_n;
}

// ----------------------------------------------------------- launchers
// All launchers assume validated arguments and return LSX_OK or
// LSX_ERR_LAUNCH.

// O/LSE merge of two partials (attn_merge).
int launch_merge(const lsx_tensor& oa, const lsx_tensor& la,
                 const lsx_tensor& ob, const lsx_tensor& lb,
                 const lsx_tensor& oo, const lsx_tensor& lo,
                 const DeviceCtx& ctx, cudaStream_t s);

// One-pass merge of n_parts partials (attn_tree_merge).
int launch_tree_merge(const lsx_tensor& op, int64_t pso, const lsx_tensor& lp,
                      int64_t psl, int n_parts, const lsx_tensor& oo,
                      const lsx_tensor& lo, const DeviceCtx& ctx,
                      cudaStream_t s);

// delta[b,h,n] = <dO[b,h,n,:], O[b,h,n,:]> into a dense f32 [B*H*N] buffer.
// With rows non-NULL it also writes the per-row statistics operand of the
// tensor-core dK/dV kernel (see RowStats) from the same row and lse.
struct RowStats {
  void* rows = nullptr;  // bf16 [B*H*N][8]
  void* ones = nullptr;  // bf16 [2][128][8] selector tiles
};
int launch_row_dot(const lsx_tensor& o, const lsx_tensor& d_o, float* delta,
                   const RowStats& stats, const lsx_tensor* lse, float scale,
                   const DeviceCtx& ctx, cudaStream_t s);

// Writes O = 0 and LSE = -inf for every row (a pair with no visible key);
// with accumulate the outputs are left as they are (the merge identity).
int launch_fill_empty(const lsx_tensor& o, const lsx_tensor& lse,
                      const DeviceCtx& ctx, cudaStream_t s);

// Zero a [B,H,N,D] view (used for gradients of keys nobody sees).
int launch_zero(const lsx_tensor& t, const DeviceCtx& ctx, cudaStream_t s);

// fp32 CUDA-core path (f32 inputs).
int launch_simt_fwd(const lsx_tensor& q, const lsx_tensor& k,
                    const lsx_tensor& v, int64_t q_off, int64_t kv_off,
                    int causal, float scale, const lsx_tensor& o,
                    const lsx_tensor& lse, int accumulate, const DeviceCtx& ctx,
                    cudaStream_t s);
int launch_simt_bwd(const lsx_tensor& q, const lsx_tensor& k,
                    const lsx_tensor& v, const lsx_tensor& lse,
                    const lsx_tensor& d_o, const float* delta, int64_t q_off,
                    int64_t kv_off, int causal, float scale,
                    const lsx_tensor& dq, const lsx_tensor& dk,
                    const lsx_tensor& dv, int accumulate, const DeviceCtx& ctx,
                    cudaStream_t s);

// Block-sparse work lists (block_sparse.cu), int32 in device memory, built
// from a block mask [n_qb][n_kb] (uint8, 128 x 128 blocks, nonzero = visible)
// ANDed with the causal rule (positions counted from 0 on both sides):
//   pair: for query-tile pair p (tiles 2p, 2p+1), the key tiles visible to
//         either tile, ascending (stride n_kb);
//   row:  for query tile i, its visible key tiles (stride n_kb);
//   col:  for key tile j, the query tiles that see it (stride n_qb).
struct BlockLists {
  const uint8_t* mask = nullptr;
  int64_t n_qb = 0, n_kb = 0;
  const int32_t* pair_count = nullptr;
  const int32_t* pair_list = nullptr;
  const int32_t* row_count = nullptr;
  const int32_t* row_list = nullptr;
  const int32_t* col_count = nullptr;
  const int32_t* col_list = nullptr;
};
size_t block_lists_bytes(int64_t lq, int64_t lk);
int build_block_lists(const uint8_t* mask, int64_t lq, int64_t lk, int causal, void* ws,
                      BlockLists* out, const DeviceCtx& ctx, cudaStream_t s);

// tcgen05 tensor-core forward (bf16 inputs).  vt: NULL (V read as stored,
// d-contiguous) or fwd_tc_workspace_bytes(v) of scratch that receives a
// key-contiguous copy of V first, which the P.V product reads faster.
size_t fwd_tc_workspace_bytes(const lsx_tensor& v);
// With bl non-NULL, each item visits only the key tiles of its block lists.
int launch_fwd_tc(const lsx_tensor& q, const lsx_tensor& k,
                  const lsx_tensor& v, int64_t q_off, int64_t kv_off,
                  int causal, float scale, const lsx_tensor& o,
                  const lsx_tensor& lse, int accumulate, void* vt,
                  const DeviceCtx& ctx, cudaStream_t s, const BlockLists* bl = nullptr);

// tcgen05 tensor-core backward (bf16 inputs).  Unless the deterministic
// mode is set, one kernel computes dK, dV and dQ (D = 128 or 64), adding each
// key tile's dQ contribution into an fp32 accumulator: copies.dq_acc
// (at D = 128 transposed [B, Hq, 128, Np], at D = 64 dense [B, Hq, Lq, 64];
// zeroed and converted to dq by the launcher) or,
// when dq itself is f32, dq directly.  Otherwise two kernels own their
// outputs: with copies.kt non-NULL, a key-contiguous copy of K is written
// there first and the dQ product reads it K-major; with NULL the K tiles
// are read as stored (MN-major), which needs no scratch beyond delta.  With
// copies.stats.rows non-NULL (written by launch_row_dot beforehand) the
// dK/dV kernel takes -LSE/scale and -delta into its score products as one
// extra rank-1 K step instead of applying them per element.  kt and dq_acc
// share one scratch region; a launch uses at most one of them.
struct BwdCopies {
  void* kt = nullptr;
  float* dq_acc = nullptr;
  RowStats stats;
};
size_t bwd_tc_copies_bytes(const lsx_tensor& q, const lsx_tensor& k);
BwdCopies bwd_tc_copies(const lsx_tensor& q, const lsx_tensor& k, void* base);
int launch_bwd_tc(const lsx_tensor& q, const lsx_tensor& k,
                  const lsx_tensor& v, const lsx_tensor& lse,
                  const lsx_tensor& d_o, const float* delta,
                  const BwdCopies& copies, int64_t q_off, int64_t kv_off,
                  int causal, float scale, const lsx_tensor& dq,
                  const lsx_tensor& dk, const lsx_tensor& dv, int accumulate,
                  const DeviceCtx& ctx, cudaStream_t s, const BlockLists* bl = nullptr);

// Split-KV decode partials (bf16 inputs, D = 128): chunk c of the cache
// writes partial block part0 + c, [parts][B * Hq][D] and [parts][B * Hq].
int launch_decode_partials(const lsx_tensor& q, const lsx_tensor& kc,
                           const lsx_tensor& vc, int64_t chunk_len,
                           float scale, float* part_o, float* part_lse,
                           const DeviceCtx& ctx, cudaStream_t s, int64_t part0 = 0);
// The same against one cache (batch 1) shared by all B query batches, read
// once per group of branches.
int launch_decode_shared(const lsx_tensor& q, const lsx_tensor& kc, const lsx_tensor& vc,
                         int64_t chunk_len, float scale, float* part_o, float* part_lse,
                         const DeviceCtx& ctx, cudaStream_t s, int64_t part0);

// Host-side forward work schedule shared with the forward kernel: the
// order in which work items are handed to persistent CTAs.
struct FwdSchedule {
  int64_t n_items;   // (B * H) * n_qpairs
  int64_t n_qpairs;  // ceil(Lq / 256)
  int64_t bh;        // B * H
};

// KV tiles of 128 keys that query tile t (rows [128 t, 128 t + 128)) must
// visit.  Shared by host (schedule statistics) and device.
__host__ __device__ inline int64_t fwd_kv_tiles(int64_t t, int64_t Lq,
                                                int64_t Lk, int64_t q_off,
                                                int64_t kv_off, int causal) {
  const int64_t r0 = t * 128;
  if (r0 >= Lq) return 0;
  int64_t kmax = Lk;
  if (causal) {
    const int64_t last = (r0 + 127 < Lq - 1 ? r0 + 127 : Lq - 1);
    const int64_t vis = q_off + last - kv_off + 1;  // keys visible to last row
    kmax = vis < Lk ? vis : Lk;
  }
  return kmax > 0 ? (kmax + 127) / 128 : 0;
}

// Work item -> (rank, bh) for the persistent grids.  The units of one
// (batch, head) pair -- query tiles or key tiles -- are ranked by cost, rank 0
// being the most expensive.  Items are grouped in bands of band_width ranks:
// band 0 holds ranks [0, W) of every (b, h), (b, h) by (b, h), then band 1,
// and so on.  Neighbouring items, which run at the same time on neighbouring
// CTAs, then share a head and stream the same K/V (or Q/dO) tiles, so most
// tile loads hit L2; and the bands still run from the most expensive ranks
// to the cheapest, which the longest-first deal below relies on.  Small
// problems (fewer than 256 units) use W = 1: plain longest-first order.
__host__ __device__ inline int64_t band_width(int64_t n_units) {
  return n_units >= 256 ? 64 : 1;
}
__host__ __device__ inline void banded_item(int64_t it, int64_t n_units, int64_t bh_n,
                                            int64_t* rank, int64_t* bh) {
  const int64_t w = band_width(n_units);
  const int64_t full = n_units / w;  // complete bands
  const int64_t per_band = w * bh_n;
  if (it < full * per_band) {
    const int64_t k = it % per_band;
    *bh = k / w;
    *rank = (it / per_band) * w + k % w;
  } else {
    const int64_t k = it - full * per_band;
    const int64_t tail = n_units - full * w;
    *bh = k / tail;
    *rank = full * w + k % tail;
  }
}

// Item index for CTA c of G in round r.  Items are in (banded) decreasing-
// cost order; CTA c takes item r*G + c on even rounds and r*G + (G-1-c) on
// odd rounds (a "snake" deal that evens out the longest-first order).
__host__ __device__ inline int64_t snake_item(int64_t c, int64_t r, int64_t G) {
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

}  // namespace lsx
