// merge.cu -- bandwidth-bound kernels: the pairwise LSE merge, the one-pass
// k-way merge, the backward row dot product and small fills.
//
// Merge rule (BurstAttention abstract: local results aggregated into global
// ones; Lean Attention abstract: online softmax is associative, so the
// combination is a reduction; Tree Attention abstract: the reduction across
// the sequence axis is a tree reduction):
//   m = max_p LSE_p,  w_p = exp(LSE_p - m),  LSE = m + log sum_p w_p,
//   O = sum_p (w_p / sum w) O_p;   all LSE_p = -inf  ->  O = 0, LSE = -inf.
//
// Layout: one warp per row of D elements; lane l owns elements
// [l*E, l*E + E) with E = D / 32, so each row is one fully coalesced access
// per tensor.  Grids are sized in multiples of the SM count.
#include <cuda_bf16.h>
#include <math.h>

#include "fwd_split.h"
#include "internal.h"

namespace lsx {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();

template <int E>
struct Vec {
  float v[E];
};

template <int E>
__device__ __forceinline__ Vec<E> load_row(const void* base, int dtype,
                                           int64_t off, int lane) {
  Vec<E> r;
  if (dtype == LSX_F32) {
    const float* p = static_cast<const float*>(base) + off + lane * E;
    if constexpr (E == 4) {
      float4 x = __ldcs(reinterpret_cast<const float4*>(p));
      r.v[0] = x.x; r.v[1] = x.y; r.v[2] = x.z; r.v[3] = x.w;
    } else if constexpr (E == 2) {
      float2 x = __ldcs(reinterpret_cast<const float2*>(p));
      r.v[0] = x.x; r.v[1] = x.y;
    } else {
      for (int e = 0; e < E; ++e) r.v[e] = p[e];
    }
  } else {
    const __nv_bfloat16* p =
        static_cast<const __nv_bfloat16*>(base) + off + lane * E;
    if constexpr (E == 4) {
      uint2 x = __ldcs(reinterpret_cast<const uint2*>(p));
      __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&x.x);
      __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&x.y);
      r.v[0] = __low2float(a); r.v[1] = __high2float(a);
      r.v[2] = __low2float(b); r.v[3] = __high2float(b);
    } else if constexpr (E == 2) {
      uint32_t x = __ldcs(reinterpret_cast<const unsigned int*>(p));
      __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&x);
      r.v[0] = __low2float(a); r.v[1] = __high2float(a);
    } else {
      for (int e = 0; e < E; ++e) r.v[e] = __bfloat162float(p[e]);
    }
  }
  return r;
}

template <int E>
__device__ __forceinline__ void store_row(void* base, int dtype, int64_t off,
                                          int lane, const Vec<E>& r) {
  if (dtype == LSX_F32) {
    float* p = static_cast<float*>(base) + off + lane * E;
    if constexpr (E == 4) {
      __stcs(reinterpret_cast<float4*>(p),
             make_float4(r.v[0], r.v[1], r.v[2], r.v[3]));
    } else if constexpr (E == 2) {
      __stcs(reinterpret_cast<float2*>(p), make_float2(r.v[0], r.v[1]));
    } else {
      for (int e = 0; e < E; ++e) p[e] = r.v[e];
    }
  } else {
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + off + lane * E;
    if constexpr (E == 4) {
      __nv_bfloat162 a = __floats2bfloat162_rn(r.v[0], r.v[1]);
      __nv_bfloat162 b = __floats2bfloat162_rn(r.v[2], r.v[3]);
      uint2 x;
      x.x = *reinterpret_cast<uint32_t*>(&a);
      x.y = *reinterpret_cast<uint32_t*>(&b);
      __stcs(reinterpret_cast<uint2*>(p), x);
    } else if constexpr (E == 2) {
      __nv_bfloat162 a = __floats2bfloat162_rn(r.v[0], r.v[1]);
      __stcs(reinterpret_cast<unsigned int*>(p),
             *reinterpret_cast<unsigned int*>(&a));
    } else {
      for (int e = 0; e < E; ++e) p[e] = __float2bfloat16_rn(r.v[e]);
    }
  }
}

struct RowIdx {
  int64_t H, N;
  __device__ __forceinline__ void split(int64_t row, int64_t& b, int64_t& h,
                                        int64_t& n) const {
    if (row < (int64_t{1} << 31) && N < (int64_t{1} << 31) && H < (int64_t{1} << 31)) {
      // 32-bit divisions where everything fits (a 64-bit one costs several
      // times as many instructions, per row of every merge)
      const uint32_t r = static_cast<uint32_t>(row), nn = static_cast<uint32_t>(N),
                     hh = static_cast<uint32_t>(H);
      const uint32_t bh = r / nn;
      n = r - bh * nn;
      const uint32_t bb = bh / hh;
      h = bh - bb * hh;
      b = bb;
      return;
    }
    n = row % N;
    const int64_t bh = row / N;
    h = bh % H;
    b = bh / H;
  }
};

// ------------------------------------------------------------ pairwise
template <int E>
__device__ __forceinline__ void merge_one(const Vec<E>& va, const Vec<E>& vb, float xa, float xb,
                                          Vec<E>& out, float& l) {
  const float m = fmaxf(xa, xb);
  if (m == kNegInf) {
    for (int e = 0; e < E; ++e) out.v[e] = 0.f;
    l = kNegInf;
  } else {
    const float wa = expf(xa - m), wb = expf(xb - m);
    const float tot = wa + wb;
    const float ra = wa / tot, rb = wb / tot;
    for (int e = 0; e < E; ++e) out.v[e] = ra * va.v[e] + rb * vb.v[e];
    l = m + logf(tot);
  }
}

// One warp per row (any layout and dtype; the dense fp32 case below is
// faster).
template <int E>
__global__ void __launch_bounds__(256) merge_kernel(
    lsx_tensor oa, lsx_tensor la, lsx_tensor ob, lsx_tensor lb, lsx_tensor oo,
    lsx_tensor lo, int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const RowIdx ri{oa.H, oa.N};
  const float* pla = static_cast<const float*>(la.data);
  const float* plb = static_cast<const float*>(lb.data);
  float* plo = static_cast<float*>(lo.data);
  for (int64_t row = w0; row < rows; row += nw) {
    int64_t b, h, n;
    ri.split(row, b, h, n);
    const float xa = pla[view_off(la, b, h, n)];
    const float xb = plb[view_off(lb, b, h, n)];
    const Vec<E> va = load_row<E>(oa.data, oa.dtype, view_off(oa, b, h, n), lane);
    const Vec<E> vb = load_row<E>(ob.data, ob.dtype, view_off(ob, b, h, n), lane);
    Vec<E> out;
    float l;
    merge_one<E>(va, vb, xa, xb, out, l);
    // all lanes have read their inputs before any store (outputs may alias)
    __syncwarp();
    store_row<E>(oo.data, oo.dtype, view_off(oo, b, h, n), lane, out);
    if (lane == 0) plo[view_off(lo, b, h, n)] = l;
  }
}

// Dense fp32 form (every O tensor [B, H, N, D] contiguous, LSE [B, H, N]
// contiguous, the output LSE separate from the inputs'): a grid-stride loop
// over 16-byte pieces, four per thread per iteration, each piece combined
// with its row's two LSE values.  A thread writes only the pieces it read,
// so the output O may be one of the inputs.
// D4: 16-byte pieces per row (D / 4), a constant so that the row of a piece
// is a shift.
template <int D4>
__global__ void __launch_bounds__(256) merge_dense_kernel(
    const float4* __restrict__ oa, const float* __restrict__ la, const float4* __restrict__ ob,
    const float* __restrict__ lb, float4* oo, float* lo, int64_t n4) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n4;
       i0 += 4 * stride) {
    float4 xa[4], xb[4];
    float sa[4], sb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n4) {
        const int64_t row = i / D4;
        xa[u] = __ldcs(oa + i);
        xb[u] = __ldcs(ob + i);
        sa[u] = __ldg(la + row);
        sb[u] = __ldg(lb + row);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < n4) {
        const float m = fmaxf(sa[u], sb[u]);
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        float l = kNegInf;
        if (m != kNegInf) {
          const float wa = expf(sa[u] - m), wb = expf(sb[u] - m);
          const float tot = wa + wb;
          const float ra = wa / tot, rb = wb / tot;
          r = make_float4(ra * xa[u].x + rb * xb[u].x, ra * xa[u].y + rb * xb[u].y,
                          ra * xa[u].z + rb * xb[u].z, ra * xa[u].w + rb * xb[u].w);
          l = m + logf(tot);
        }
        __stcs(oo + i, r);
        if (i % D4 == 0) lo[i / D4] = l;
      }
    }
  }
}

// ------------------------------------------------------------- k-way
// One warp per row (n_parts <= 32).  Lane p holds partial p's LSE; the
// partial rows are read four at a time, loads first, and accumulated in the
// order p = 0, 1, ..., n-1, so the result does not depend on the launch shape.
template <int E>
__global__ void __launch_bounds__(256) tree_merge_warp_kernel(
    lsx_tensor op, int64_t pso, lsx_tensor lp, int64_t psl, int n_parts,
    lsx_tensor oo, lsx_tensor lo, int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const RowIdx ri{op.H, op.N};
  const float* plp = static_cast<const float*>(lp.data);
  for (int64_t row = w0; row < rows; row += nw) {
    int64_t b, h, n;
    ri.split(row, b, h, n);
    const int64_t lbase = view_off(lp, b, h, n);
    const int64_t obase = view_off(op, b, h, n);
    const float x = lane < n_parts ? plp[lbase + lane * psl] : kNegInf;
    float m = x;
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    const float wl = (m == kNegInf || lane >= n_parts) ? 0.f : expf(x - m);
    float tot = wl;
    for (int s = 16; s > 0; s >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, s);
    Vec<E> acc;
    for (int e = 0; e < E; ++e) acc.v[e] = 0.f;
    if (m != kNegInf) {
      for (int p0 = 0; p0 < n_parts; p0 += 4) {
        Vec<E> xs[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (p0 + u < n_parts) xs[u] = load_row<E>(op.data, op.dtype, obase + (p0 + u) * pso, lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = __shfl_sync(0xffffffffu, wl, (p0 + u) & 31);
          if (p0 + u < n_parts)
            for (int e = 0; e < E; ++e) acc.v[e] = fmaf(w, xs[u].v[e], acc.v[e]);
        }
      }
      const float inv = 1.f / tot;
      for (int e = 0; e < E; ++e) acc.v[e] *= inv;
    }
    store_row<E>(oo.data, oo.dtype, view_off(oo, b, h, n), lane, acc);
    if (lane == 0 && lo.data != nullptr)
      static_cast<float*>(lo.data)[view_off(lo, b, h, n)] =
          (m == kNegInf) ? kNegInf : m + logf(tot);
  }
}

// The pieces of split rows (FwdSplit): one warp per row, lane p holding
// piece p's LSE.  A row has as many pieces as its query pair: ceil(its
// pair's visible key tiles / piece_w), from the same causal geometry the
// forward used; slot p of the partials sits p * B * H * Lq rows on.  Pieces
// are combined in the order p = 0, 1, ..., like tree_merge_warp_kernel.
template <int E>
__global__ void __launch_bounds__(256) merge_pieces_kernel(
    const float* __restrict__ part_o, const float* __restrict__ part_lse, int64_t piece_w,
    int64_t Lk, int64_t q_off, int64_t kv_off, int causal, lsx_tensor oo, lsx_tensor lo,
    int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const RowIdx ri{oo.H, oo.N};
  for (int64_t row = w0; row < rows; row += nw) {
    int64_t b, h, n;
    ri.split(row, b, h, n);
    const int64_t pair = (n / 128) / 2;
    const int64_t t0 = fwd_kv_tiles(2 * pair, oo.N, Lk, q_off, kv_off, causal);
    const int64_t t1 = fwd_kv_tiles(2 * pair + 1, oo.N, Lk, q_off, kv_off, causal);
    const int64_t tiles = t0 > t1 ? t0 : t1;
    const int n_parts = static_cast<int>((tiles + piece_w - 1) / piece_w);
    const float x = lane < n_parts ? part_lse[lane * rows + row] : kNegInf;
    float m = x;
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    const float wl = (m == kNegInf || lane >= n_parts) ? 0.f : expf(x - m);
    float tot = wl;
    for (int s = 16; s > 0; s >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, s);
    Vec<E> acc;
    for (int e = 0; e < E; ++e) acc.v[e] = 0.f;
    if (m != kNegInf) {
      for (int p0 = 0; p0 < n_parts; p0 += 4) {
        Vec<E> xs[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (p0 + u < n_parts)
            xs[u] = load_row<E>(part_o, LSX_F32, ((p0 + u) * rows + row) * (32 * E), lane);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = __shfl_sync(0xffffffffu, wl, (p0 + u) & 31);
          if (p0 + u < n_parts)
            for (int e = 0; e < E; ++e) acc.v[e] = fmaf(w, xs[u].v[e], acc.v[e]);
        }
      }
      const float inv = 1.f / tot;
      for (int e = 0; e < E; ++e) acc.v[e] *= inv;
    }
    store_row<E>(oo.data, oo.dtype, view_off(oo, b, h, n), lane, acc);
    if (lane == 0)
      static_cast<float*>(lo.data)[view_off(lo, b, h, n)] =
          (m == kNegInf) ? kNegInf : m + logf(tot);
  }
}

// One block of 8 warps per row for many partials: warp w takes partials
// p = w, w + 8, ...; the 8 warp sums are combined in warp order.
template <int E>
__global__ void __launch_bounds__(256) tree_merge_block_kernel(
    lsx_tensor op, int64_t pso, lsx_tensor lp, int64_t psl, int n_parts,
    lsx_tensor oo, lsx_tensor lo, int64_t rows) {
  __shared__ float s_max[8];
  __shared__ float s_tot[8];
  __shared__ float s_acc[8][32 * E];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const RowIdx ri{op.H, op.N};
  const float* plp = static_cast<const float*>(lp.data);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    int64_t b, h, n;
    ri.split(row, b, h, n);
    const int64_t lbase = view_off(lp, b, h, n);
    const int64_t obase = view_off(op, b, h, n);
    float m = kNegInf;
    for (int p = threadIdx.x; p < n_parts; p += blockDim.x)
      m = fmaxf(m, plp[lbase + p * psl]);
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    if (lane == 0) s_max[warp] = m;
    __syncthreads();
    m = s_max[0];
    for (int w = 1; w < 8; ++w) m = fmaxf(m, s_max[w]);
    Vec<E> acc;
    for (int e = 0; e < E; ++e) acc.v[e] = 0.f;
    float tot = 0.f;
    if (m != kNegInf) {
      for (int p = warp; p < n_parts; p += 8) {
        const float w = expf(plp[lbase + p * psl] - m);
        const Vec<E> x = load_row<E>(op.data, op.dtype, obase + p * pso, lane);
        tot += w;
        for (int e = 0; e < E; ++e) acc.v[e] = fmaf(w, x.v[e], acc.v[e]);
      }
    }
    for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc.v[e];
    if (lane == 0) s_tot[warp] = tot;
    __syncthreads();
    if (warp == 0) {
      Vec<E> out;
      float t = 0.f;
      for (int e = 0; e < E; ++e) out.v[e] = 0.f;
      for (int w = 0; w < 8; ++w) {
        t += s_tot[w];
        for (int e = 0; e < E; ++e) out.v[e] += s_acc[w][lane * E + e];
      }
      if (m != kNegInf) {
        const float inv = 1.f / t;
        for (int e = 0; e < E; ++e) out.v[e] *= inv;
      }
      store_row<E>(oo.data, oo.dtype, view_off(oo, b, h, n), lane, out);
      if (lane == 0 && lo.data != nullptr)
        static_cast<float*>(lo.data)[view_off(lo, b, h, n)] =
            (m == kNegInf) ? kNegInf : m + logf(t);
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------- row dot
// bf16 bits of x rounded to nearest, and the f32 remainder x - that value
// (exact: the remainder of a round to 8 significant bits fits in f32).
__device__ __forceinline__ uint32_t bf16_split(float x, float& rem) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  rem = x - __bfloat162float(h);
  return static_cast<uint32_t>(__bfloat16_as_ushort(h));
}

// Row statistics operand of the tensor-core dK/dV kernel, one 16-byte row per
// query row: bf16 {c1, c2, c3, d1, d2, d3, 0, 0} with c1 + c2 + c3 = c / 2,
// c = -LSE / scale (c = -2^100 when LSE = -inf, so that the row's
// probabilities underflow to 0), and d1 + d2 + d3 = -delta / 2: each value
// is carried by three bf16 terms (24 significant bits).  The halving is
// undone by the kernel, which reads the 8 stored columns twice in its K step
// of 16.  Selector tiles: rows of {1, 1, 1, 0, 0, 0, 0, 0} (tile 0) and
// {0, 0, 0, 1, 1, 1, 0, 0} (tile 1), so that a K step of
// (selector x statistics^T) adds c or -delta to every score of a query
// column.
__device__ __forceinline__ uint4 row_stats(float lse, float delta, float inv_scale) {
  const float c = lse == kNegInf ? -0x1p100f : -lse * inv_scale;
  float r;
  const uint32_t c1 = bf16_split(0.5f * c, r);
  const uint32_t c2 = bf16_split(r, r);
  const uint32_t c3 = bf16_split(r, r);
  const uint32_t d1 = bf16_split(-0.5f * delta, r);
  const uint32_t d2 = bf16_split(r, r);
  const uint32_t d3 = bf16_split(r, r);
  return make_uint4(c1 | (c2 << 16), c3 | (d1 << 16), d2 | (d3 << 16), 0u);
}

template <int E>
__global__ void __launch_bounds__(256) row_dot_kernel(lsx_tensor o,
                                                      lsx_tensor d_o,
                                                      float* delta,
                                                      int64_t rows,
                                                      uint4* stats,
                                                      uint4* ones,
                                                      lsx_tensor lse,
                                                      float inv_scale) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const RowIdx ri{o.H, o.N};
  if (ones != nullptr && blockIdx.x == 0) {
    const uint32_t one = 0x3F80u;  // bf16 1.0
    ones[threadIdx.x] = threadIdx.x < 128
                            ? make_uint4(one | (one << 16), one, 0u, 0u)
                            : make_uint4(0u, one << 16, one | (one << 16), 0u);
  }
  for (int64_t row = w0; row < rows; row += nw) {
    int64_t b, h, n;
    ri.split(row, b, h, n);
    const Vec<E> x = load_row<E>(o.data, o.dtype, view_off(o, b, h, n), lane);
    const Vec<E> y = load_row<E>(d_o.data, d_o.dtype, view_off(d_o, b, h, n), lane);
    float s = 0.f;
    for (int e = 0; e < E; ++e) s = fmaf(x.v[e], y.v[e], s);
    for (int k = 16; k > 0; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
    if (lane == 0) {
      delta[row] = s;
      if (stats != nullptr)
        stats[row] = row_stats(static_cast<const float*>(lse.data)[view_off(lse, b, h, n)], s,
                               inv_scale);
    }
  }
}

// -------------------------------------------------------------- fills
template <int E>
__global__ void __launch_bounds__(256) fill_kernel(lsx_tensor o,
                                                   lsx_tensor lse,
                                                   int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const RowIdx ri{o.H, o.N};
  Vec<E> z;
  for (int e = 0; e < E; ++e) z.v[e] = 0.f;
  for (int64_t row = w0; row < rows; row += nw) {
    int64_t b, h, n;
    ri.split(row, b, h, n);
    store_row<E>(o.data, o.dtype, view_off(o, b, h, n), lane, z);
    if (lane == 0 && lse.data != nullptr)
      static_cast<float*>(lse.data)[view_off(lse, b, h, n)] = kNegInf;
  }
}

// Grid of a row-loop kernel of 256-thread blocks: one block per `per_block`
// rows, capped at the blocks the GPU holds at once (SMs x resident blocks per
// SM for this kernel), so that every block is resident and the grid-stride
// loops share the rows evenly instead of leaving a partial second wave.
template <typename Kernel>
int grid_for_rows(Kernel kernel, int64_t rows, const DeviceCtx& ctx, int64_t per_block) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t blocks = ceil_div(rows, per_block);
  const int64_t cap = static_cast<int64_t>(ctx.sm_count) * per_sm;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

bool dense_rows(const lsx_tensor& t) {
  return t.stride_n == t.D && t.stride_h == t.N * t.D && (t.B == 1 || t.stride_b == t.H * t.N * t.D);
}
bool dense_lse(const lsx_tensor& t) {
  return t.stride_n == 1 && t.stride_h == t.N && (t.B == 1 || t.stride_b == t.H * t.N);
}
// Whether two dense [B, H, N, D] fp32 views share any byte.
bool overlaps(const lsx_tensor& a, const lsx_tensor& b) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.data), b0 = reinterpret_cast<uintptr_t>(b.data);
  const uintptr_t an = static_cast<uintptr_t>(a.B * a.H * a.N * a.D) * 4;
  const uintptr_t bn = static_cast<uintptr_t>(b.B * b.H * b.N * b.D) * 4;
  return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

#define LSX_DISPATCH_E(D, ...)                     \
  switch (D) {                                     \
    case 128: { constexpr int E = 4; __VA_ARGS__; break; } \
    case 64: { constexpr int E = 2; __VA_ARGS__; break; }  \
    default: return LSX_ERR_UNSUPPORTED;           \
  }

int launch_merge(const lsx_tensor& oa, const lsx_tensor& la,
                 const lsx_tensor& ob, const lsx_tensor& lb,
                 const lsx_tensor& oo, const lsx_tensor& lo,
                 const DeviceCtx& ctx, cudaStream_t s) {
  const int64_t rows = oa.B * oa.H * oa.N;
  if (rows == 0) return LSX_OK;
  timing_begin(kKidMerge, s);
  const bool dense = oa.dtype == LSX_F32 && ob.dtype == LSX_F32 && oo.dtype == LSX_F32 &&
                     dense_rows(oa) && dense_rows(ob) && dense_rows(oo) && dense_lse(la) &&
                     dense_lse(lb) && dense_lse(lo) && oa.D % 4 == 0 &&
                     (oo.data == oa.data || oo.data == ob.data ||
                      (!overlaps(oo, oa) && !overlaps(oo, ob))) &&
                     lo.data != la.data && lo.data != lb.data;
  if (dense) {
    const int64_t n4 = rows * oa.D / 4;
    auto kern = oa.D == 128 ? merge_dense_kernel<32> : merge_dense_kernel<16>;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    const int64_t need = ceil_div(n4, 256 * 4);
    const int64_t cap = static_cast<int64_t>(ctx.sm_count) * per_sm;
    kern<<<static_cast<int>(need < cap ? need : cap), 256, 0, s>>>(
        static_cast<const float4*>(oa.data), static_cast<const float*>(la.data),
        static_cast<const float4*>(ob.data), static_cast<const float*>(lb.data),
        static_cast<float4*>(oo.data), static_cast<float*>(lo.data), n4);
    timing_end(kKidMerge, s);
    return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
  }
  LSX_DISPATCH_E(oa.D, merge_kernel<E><<<grid_for_rows(merge_kernel<E>, rows, ctx, 8), 256, 0,
                                          s>>>(oa, la, ob, lb, oo, lo, rows));
  timing_end(kKidMerge, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

int launch_tree_merge(const lsx_tensor& op, int64_t pso, const lsx_tensor& lp,
                      int64_t psl, int n_parts, const lsx_tensor& oo,
                      const lsx_tensor& lo, const DeviceCtx& ctx,
                      cudaStream_t s) {
  const int64_t rows = op.B * op.H * op.N;
  if (rows == 0) return LSX_OK;
  timing_begin(kKidTreeMerge, s);
  if (n_parts <= 16) {
    LSX_DISPATCH_E(op.D, tree_merge_warp_kernel<E><<<
                             grid_for_rows(tree_merge_warp_kernel<E>, rows, ctx, 8), 256, 0, s>>>(
                             op, pso, lp, psl, n_parts, oo, lo, rows));
  } else {
    LSX_DISPATCH_E(op.D, tree_merge_block_kernel<E><<<
                             grid_for_rows(tree_merge_block_kernel<E>, rows, ctx, 1), 256, 0, s>>>(
                             op, pso, lp, psl, n_parts, oo, lo, rows));
  }
  timing_end(kKidTreeMerge, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

int launch_merge_pieces(const FwdSplit& split, int64_t q_off, int64_t kv_off, int causal,
                        int64_t Lk, const lsx_tensor& o, const lsx_tensor& lse,
                        const DeviceCtx& ctx, cudaStream_t s) {
  const int64_t rows = o.B * o.H * o.N;
  if (rows == 0) return LSX_OK;
  if (split.piece_w <= 0 || split.kmax < 1 || split.kmax > 32) return LSX_ERR_UNSUPPORTED;
  timing_begin(kKidTreeMerge, s);
  LSX_DISPATCH_E(o.D, merge_pieces_kernel<E><<<grid_for_rows(merge_pieces_kernel<E>, rows, ctx, 8),
                                                256, 0, s>>>(split.part_o, split.part_lse,
                                                             split.piece_w, Lk, q_off, kv_off,
                                                             causal, o, lse, rows));
  timing_end(kKidTreeMerge, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

int launch_row_dot(const lsx_tensor& o, const lsx_tensor& d_o, float* delta,
                   const RowStats& stats, const lsx_tensor* lse, float scale,
                   const DeviceCtx& ctx, cudaStream_t s) {
  const int64_t rows = o.B * o.H * o.N;
  if (rows == 0) return LSX_OK;
  uint4* st = static_cast<uint4*>(stats.rows);
  uint4* on = static_cast<uint4*>(stats.ones);
  lsx_tensor l{};
  if (st != nullptr) {
    if (lse == nullptr || on == nullptr) return LSX_ERR_LAUNCH;
    l = *lse;
  }
  const float inv_scale = static_cast<float>(1.0 / static_cast<double>(scale));
  timing_begin(kKidRowDot, s);
  LSX_DISPATCH_E(o.D, row_dot_kernel<E><<<grid_for_rows(row_dot_kernel<E>, rows, ctx, 8), 256, 0,
                                            s>>>(o, d_o, delta, rows, st, on, l, inv_scale));
  timing_end(kKidRowDot, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

int launch_fill_empty(const lsx_tensor& o, const lsx_tensor& lse,
                      const DeviceCtx& ctx, cudaStream_t s) {
  const int64_t rows = o.B * o.H * o.N;
  if (rows == 0) return LSX_OK;
  timing_begin(kKidFill, s);
  LSX_DISPATCH_E(o.D, fill_kernel<E><<<grid_for_rows(fill_kernel<E>, rows, ctx, 8), 256, 0, s>>>(
                          o, lse, rows));
  timing_end(kKidFill, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

int launch_zero(const lsx_tensor& t, const DeviceCtx& ctx, cudaStream_t s) {
  lsx_tensor none = t;
  none.data = nullptr;
  return launch_fill_empty(t, none, ctx, s);
}

}  // namespace lsx
