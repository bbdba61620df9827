// block_sparse.cu -- work lists for block-sparse attention (the Fine-grained
// Attention I/O Complexity page, abstract: the analysis extends to sparse
// attention; the BriefGPT BurstAttention page's related work: FlashAttention
// extended to a broad class of sparsity patterns).
//
// A block mask [n_qb][n_kb] of 128 x 128 blocks (uint8, nonzero = the block's
// scores exist), ANDed with the causal rule, becomes three compacted lists
// that the persistent kernels walk instead of the dense tile ranges: per
// query-tile pair (forward), per query tile (dQ) and per key tile (dK/dV).
// One warp per list: ballot over 32 candidates at a time, prefix popcount for
// the slot of each set entry, so every list comes out in ascending order.
#include <stdint.h>

#include "internal.h"

namespace lsx {
namespace {

struct ListLayout {
  size_t pair_count, pair_list, row_count, row_list, col_count, col_list, total;
};

inline size_t align256(size_t n) { return (n + 255) / 256 * 256; }

ListLayout list_layout(int64_t n_qb, int64_t n_kb) {
  const int64_t n_pairs = (n_qb + 1) / 2;
  ListLayout l;
  size_t off = 0;
  l.pair_count = off; off += align256(static_cast<size_t>(n_pairs) * 4);
  l.pair_list = off;  off += align256(static_cast<size_t>(n_pairs * n_kb) * 4);
  l.row_count = off;  off += align256(static_cast<size_t>(n_qb) * 4);
  l.row_list = off;   off += align256(static_cast<size_t>(n_qb * n_kb) * 4);
  l.col_count = off;  off += align256(static_cast<size_t>(n_kb) * 4);
  l.col_list = off;   off += align256(static_cast<size_t>(n_kb * n_qb) * 4);
  l.total = off;
  return l;
}

// Appends the candidates `on` of this 32-wide step to list[count ...].
__device__ __forceinline__ void append(bool on, int32_t value, int32_t* list, int32_t& count) {
  const unsigned bal = __ballot_sync(0xffffffffu, on);
  const int lane = threadIdx.x & 31;
  if (on) list[count + __popc(bal & ((1u << lane) - 1u))] = value;
  count += __popc(bal);
}

__global__ void __launch_bounds__(256) build_lists_kernel(
    const uint8_t* __restrict__ mask, int64_t n_qb, int64_t n_kb, int64_t lq, int64_t lk,
    int causal, int32_t* pair_count, int32_t* pair_list, int32_t* row_count,
    int32_t* row_list, int32_t* col_count, int32_t* col_list) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n_pairs = (n_qb + 1) / 2;
  int32_t count = 0;
  if (w < n_pairs) {
    const int64_t t0 = 2 * w, t1 = 2 * w + 1;
    const bool has1 = t1 < n_qb;
    // key tiles the pair's last query tile can see (causal), else all
    const int64_t lim =
        causal ? fwd_kv_tiles(has1 ? t1 : t0, lq, lk, 0, 0, 1) : n_kb;
    for (int64_t j0 = 0; j0 < n_kb; j0 += 32) {
      const int64_t j = j0 + lane;
      const bool on = j < lim && (mask[t0 * n_kb + j] != 0 || (has1 && mask[t1 * n_kb + j] != 0));
      append(on, static_cast<int32_t>(j), pair_list + w * n_kb, count);
    }
    if (lane == 0) pair_count[w] = count;
  } else if (w < n_pairs + n_qb) {
    const int64_t i = w - n_pairs;
    const int64_t lim = causal ? fwd_kv_tiles(i, lq, lk, 0, 0, 1) : n_kb;
    for (int64_t j0 = 0; j0 < n_kb; j0 += 32) {
      const int64_t j = j0 + lane;
      const bool on = j < lim && mask[i * n_kb + j] != 0;
      append(on, static_cast<int32_t>(j), row_list + i * n_kb, count);
    }
    if (lane == 0) row_count[i] = count;
  } else if (w < n_pairs + n_qb + n_kb) {
    const int64_t j = w - n_pairs - n_qb;
    // first query tile with a row at or after key 128 j (causal)
    int64_t ib = 0;
    if (causal) ib = 128 * j > lq - 1 ? n_qb : (128 * j) / 128;
    for (int64_t i0 = 0; i0 < n_qb; i0 += 32) {
      const int64_t i = i0 + lane;
      const bool on = i >= ib && i < n_qb && mask[i * n_kb + j] != 0;
      append(on, static_cast<int32_t>(i), col_list + j * n_qb, count);
    }
    if (lane == 0) col_count[j] = count;
  }
}

}  // namespace

size_t block_lists_bytes(int64_t lq, int64_t lk) {
  return list_layout(ceil_div(lq, 128), ceil_div(lk, 128)).total;
}

int build_block_lists(const uint8_t* mask, int64_t lq, int64_t lk, int causal, void* ws,
                      BlockLists* out, const DeviceCtx& ctx, cudaStream_t s) {
  (void)ctx;
  const int64_t n_qb = ceil_div(lq, 128), n_kb = ceil_div(lk, 128);
  const ListLayout l = list_layout(n_qb, n_kb);
  char* base = static_cast<char*>(ws);
  BlockLists b;
  b.mask = mask;
  b.n_qb = n_qb;
  b.n_kb = n_kb;
  b.pair_count = reinterpret_cast<const int32_t*>(base + l.pair_count);
  b.pair_list = reinterpret_cast<const int32_t*>(base + l.pair_list);
  b.row_count = reinterpret_cast<const int32_t*>(base + l.row_count);
  b.row_list = reinterpret_cast<const int32_t*>(base + l.row_list);
  b.col_count = reinterpret_cast<const int32_t*>(base + l.col_count);
  b.col_list = reinterpret_cast<const int32_t*>(base + l.col_list);
  *out = b;
  const int64_t warps = (n_qb + 1) / 2 + n_qb + n_kb;
  const int64_t blocks = ceil_div(warps, 8);
  if (blocks > 0x7fffffff) return LSX_ERR_UNSUPPORTED;
  timing_begin(kKidBlockLists, s);
  build_lists_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      mask, n_qb, n_kb, lq, lk, causal, reinterpret_cast<int32_t*>(base + l.pair_count),
      reinterpret_cast<int32_t*>(base + l.pair_list),
      reinterpret_cast<int32_t*>(base + l.row_count),
      reinterpret_cast<int32_t*>(base + l.row_list),
      reinterpret_cast<int32_t*>(base + l.col_count),
      reinterpret_cast<int32_t*>(base + l.col_list));
  timing_end(kKidBlockLists, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

}  // namespace lsx
