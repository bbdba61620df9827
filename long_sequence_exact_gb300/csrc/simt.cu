// simt.cu -- fp32 CUDA-core path for f32 inputs (exact attention of one
// chunk pair, forward and backward), kept in fp32 end to end so that results
// agree with an fp64 evaluation to ~1e-6.
//
// Forward: one warp per query row; lane l holds elements [l*E, l*E+E) of q,
// of the running output and of every key/value row it reads.  The online
// softmax (running max m, running sum l, output rescaled by exp(m_old -
// m_new)) follows the local attention computation of BurstAttention (method
// section) with the row state of Lean Attention's online softmax (abstract).
// Backward (DistFlashAttn core concepts: gradients from the saved output and
// LSE, no forward re-run): P_ij = exp(s_ij - LSE_i) from the saved LSE,
// dS_ij = P_ij (dP_ij - delta_i) with delta_i = <dO_i, O_i>; dQ by a warp
// per query row, dK/dV by a warp per key row (no atomics, deterministic).
#include <math.h>

#include "internal.h"

namespace lsx {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ float warp_sum(float x) {
  for (int k = 16; k > 0; k >>= 1) x += __shfl_xor_sync(0xffffffffu, x, k);
  return __shfl_sync(0xffffffffu, x, 0);  // one value for every lane
}

template <int E>
__device__ __forceinline__ void ld(const float* p, float (&x)[E]) {
  if constexpr (E == 4) {
    float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
  }
}
template <int E>
__device__ __forceinline__ void st(float* p, const float (&x)[E]) {
  if constexpr (E == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  } else {
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
  }
}

struct PairGeom {
  int64_t q_off, kv_off;
  int causal;
  // last key index (exclusive) visible to query row i
  __device__ __forceinline__ int64_t key_end(int64_t i, int64_t Lk) const {
    if (!causal) return Lk;
    int64_t e = q_off + i - kv_off + 1;
    return e < 0 ? 0 : (e < Lk ? e : Lk);
  }
  // first query row that sees key j
  __device__ __forceinline__ int64_t query_begin(int64_t j) const {
    if (!causal) return 0;
    int64_t b = kv_off + j - q_off;
    return b < 0 ? 0 : b;
  }
};

template <int E>
__global__ void __launch_bounds__(256) simt_fwd_kernel(
    lsx_tensor q, lsx_tensor k, lsx_tensor v, lsx_tensor o, lsx_tensor lse,
    PairGeom g, float scale, int accumulate) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = q.B * q.H * q.N;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t group = q.H / k.H;
  for (int64_t row = w0; row < rows; row += nw) {
    const int64_t i = row % q.N, bh = row / q.N, h = bh % q.H, b = bh / q.H;
    const int64_t hk = h / group;
    float qr[E], acc[E];
    ld<E>(static_cast<const float*>(q.data) + view_off(q, b, h, i) + lane * E, qr);
    for (int e = 0; e < E; ++e) { qr[e] *= scale; acc[e] = 0.f; }
    float m = kNegInf, l = 0.f;
    const int64_t kend = g.key_end(i, k.N);
    const float* kp = static_cast<const float*>(k.data) + view_off(k, b, hk, 0) + lane * E;
    const float* vp = static_cast<const float*>(v.data) + view_off(v, b, hk, 0) + lane * E;
    for (int64_t j = 0; j < kend; ++j) {
      float kr[E], vr[E];
      ld<E>(kp + j * k.stride_n, kr);
      float s = 0.f;
      for (int e = 0; e < E; ++e) s = fmaf(qr[e], kr[e], s);
      s = warp_sum(s);
      if (s > m) {
        const float a = expf(m - s);  // exp(-inf) = 0 on the first key
        l *= a;
        for (int e = 0; e < E; ++e) acc[e] *= a;
        m = s;
      }
      const float p = expf(s - m);
      l += p;
      ld<E>(vp + j * v.stride_n, vr);
      for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vr[e], acc[e]);
    }
    float out_l = kNegInf;
    if (l > 0.f) {
      const float inv = 1.f / l;
      for (int e = 0; e < E; ++e) acc[e] *= inv;
      out_l = m + logf(l);
    }
    float* op = static_cast<float*>(o.data) + view_off(o, b, h, i) + lane * E;
    float* lp = static_cast<float*>(lse.data) + view_off(lse, b, h, i);
    if (accumulate) {
      // merge into the partial already held in (o, lse)
      const float old_l = *lp;
      float old[E];
      ld<E>(op, old);
      const float mm = fmaxf(old_l, out_l);
      if (mm == kNegInf) {
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        out_l = kNegInf;
      } else {
        const float wa = expf(old_l - mm), wb = expf(out_l - mm);
        const float tot = wa + wb;
        for (int e = 0; e < E; ++e) acc[e] = (wa * old[e] + wb * acc[e]) / tot;
        out_l = mm + logf(tot);
      }
    }
    __syncwarp();
    st<E>(op, acc);
    if (lane == 0) *lp = out_l;
  }
}

// dQ: one warp per query row.
template <int E>
__global__ void __launch_bounds__(256) simt_dq_kernel(
    lsx_tensor q, lsx_tensor k, lsx_tensor v, lsx_tensor lse, lsx_tensor d_o,
    const float* __restrict__ delta, lsx_tensor dq, PairGeom g, float scale,
    int accumulate) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = q.B * q.H * q.N;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t group = q.H / k.H;
  for (int64_t row = w0; row < rows; row += nw) {
    const int64_t i = row % q.N, bh = row / q.N, h = bh % q.H, b = bh / q.H;
    const int64_t hk = h / group;
    float qr[E], dor[E], acc[E];
    ld<E>(static_cast<const float*>(q.data) + view_off(q, b, h, i) + lane * E, qr);
    ld<E>(static_cast<const float*>(d_o.data) + view_off(d_o, b, h, i) + lane * E, dor);
    for (int e = 0; e < E; ++e) { qr[e] *= scale; acc[e] = 0.f; }
    const float li = static_cast<const float*>(lse.data)[view_off(lse, b, h, i)];
    const float di = delta[row];
    const int64_t kend = (li == kNegInf) ? 0 : g.key_end(i, k.N);
    const float* kp = static_cast<const float*>(k.data) + view_off(k, b, hk, 0) + lane * E;
    const float* vp = static_cast<const float*>(v.data) + view_off(v, b, hk, 0) + lane * E;
    for (int64_t j = 0; j < kend; ++j) {
      float kr[E], vr[E];
      ld<E>(kp + j * k.stride_n, kr);
      ld<E>(vp + j * v.stride_n, vr);
      float s = 0.f, dp = 0.f;
      for (int e = 0; e < E; ++e) { s = fmaf(qr[e], kr[e], s); dp = fmaf(dor[e], vr[e], dp); }
      s = warp_sum(s);
      dp = warp_sum(dp);
      const float ds = expf(s - li) * (dp - di);
      for (int e = 0; e < E; ++e) acc[e] = fmaf(ds, kr[e], acc[e]);
    }
    float* out = static_cast<float*>(dq.data) + view_off(dq, b, h, i) + lane * E;
    for (int e = 0; e < E; ++e) acc[e] *= scale;
    if (accumulate) {
      float old[E];
      ld<E>(out, old);
      for (int e = 0; e < E; ++e) acc[e] += old[e];
    }
    st<E>(out, acc);
  }
}

// dK, dV: one warp per key row; sums over the query heads of its group.
template <int E>
__global__ void __launch_bounds__(256) simt_dkdv_kernel(
    lsx_tensor q, lsx_tensor k, lsx_tensor v, lsx_tensor lse, lsx_tensor d_o,
    const float* __restrict__ delta, lsx_tensor dk, lsx_tensor dv, PairGeom g,
    float scale, int accumulate) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = k.B * k.H * k.N;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t group = q.H / k.H;
  for (int64_t row = w0; row < rows; row += nw) {
    const int64_t j = row % k.N, bh = row / k.N, hk = bh % k.H, b = bh / k.H;
    float kr[E], vr[E], ak[E], av[E];
    ld<E>(static_cast<const float*>(k.data) + view_off(k, b, hk, j) + lane * E, kr);
    ld<E>(static_cast<const float*>(v.data) + view_off(v, b, hk, j) + lane * E, vr);
    for (int e = 0; e < E; ++e) { kr[e] *= scale; ak[e] = 0.f; av[e] = 0.f; }
    const int64_t ibeg = g.query_begin(j);
    for (int64_t hh = 0; hh < group; ++hh) {
      const int64_t h = hk * group + hh;
      const float* qp = static_cast<const float*>(q.data) + view_off(q, b, h, 0) + lane * E;
      const float* dop = static_cast<const float*>(d_o.data) + view_off(d_o, b, h, 0) + lane * E;
      const float* lp = static_cast<const float*>(lse.data) + view_off(lse, b, h, 0);
      const float* dl = delta + (b * q.H + h) * q.N;
      for (int64_t i = ibeg; i < q.N; ++i) {
        const float li = lp[i * lse.stride_n];
        if (li == kNegInf) continue;
        float qr[E], dor[E];
        ld<E>(qp + i * q.stride_n, qr);
        ld<E>(dop + i * d_o.stride_n, dor);
        float s = 0.f, dp = 0.f;
        for (int e = 0; e < E; ++e) { s = fmaf(qr[e], kr[e], s); dp = fmaf(dor[e], vr[e], dp); }
        s = warp_sum(s);
        dp = warp_sum(dp);
        const float p = expf(s - li);
        const float ds = p * (dp - dl[i]);
        for (int e = 0; e < E; ++e) {
          ak[e] = fmaf(ds, qr[e], ak[e]);
          av[e] = fmaf(p, dor[e], av[e]);
        }
      }
    }
    float* pk = static_cast<float*>(dk.data) + view_off(dk, b, hk, j) + lane * E;
    float* pv = static_cast<float*>(dv.data) + view_off(dv, b, hk, j) + lane * E;
    for (int e = 0; e < E; ++e) ak[e] *= scale;
    if (accumulate) {
      float ok[E], ov[E];
      ld<E>(pk, ok);
      ld<E>(pv, ov);
      for (int e = 0; e < E; ++e) { ak[e] += ok[e]; av[e] += ov[e]; }
    }
    st<E>(pk, ak);
    st<E>(pv, av);
  }
}

int grid_rows(int64_t rows, const DeviceCtx& ctx) {
  const int64_t blocks = ceil_div(rows, 8);
  const int64_t cap = static_cast<int64_t>(ctx.sm_count) * 8;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

int launch_simt_fwd(const lsx_tensor& q, const lsx_tensor& k,
                    const lsx_tensor& v, int64_t q_off, int64_t kv_off,
                    int causal, float scale, const lsx_tensor& o,
                    const lsx_tensor& lse, int accumulate, const DeviceCtx& ctx,
                    cudaStream_t s) {
  const int64_t rows = q.B * q.H * q.N;
  if (rows == 0) return LSX_OK;
  const PairGeom g{q_off, kv_off, causal};
  const int grid = grid_rows(rows, ctx);
  timing_begin(kKidSimtFwd, s);
  if (q.D == 128)
    simt_fwd_kernel<4><<<grid, 256, 0, s>>>(q, k, v, o, lse, g, scale, accumulate);
  else if (q.D == 64)
    simt_fwd_kernel<2><<<grid, 256, 0, s>>>(q, k, v, o, lse, g, scale, accumulate);
  else
    return LSX_ERR_UNSUPPORTED;
  timing_end(kKidSimtFwd, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

int launch_simt_bwd(const lsx_tensor& q, const lsx_tensor& k,
                    const lsx_tensor& v, const lsx_tensor& lse,
                    const lsx_tensor& d_o, const float* delta, int64_t q_off,
                    int64_t kv_off, int causal, float scale,
                    const lsx_tensor& dq, const lsx_tensor& dk,
                    const lsx_tensor& dv, int accumulate, const DeviceCtx& ctx,
                    cudaStream_t s) {
  const PairGeom g{q_off, kv_off, causal};
  const int64_t qrows = q.B * q.H * q.N, krows = k.B * k.H * k.N;
  if (q.D != 128 && q.D != 64) return LSX_ERR_UNSUPPORTED;
  timing_begin(kKidSimtBwd, s);
  if (qrows > 0) {
    const int grid = grid_rows(qrows, ctx);
    if (q.D == 128)
      simt_dq_kernel<4><<<grid, 256, 0, s>>>(q, k, v, lse, d_o, delta, dq, g, scale, accumulate);
    else
      simt_dq_kernel<2><<<grid, 256, 0, s>>>(q, k, v, lse, d_o, delta, dq, g, scale, accumulate);
  }
  if (krows > 0) {
    const int grid = grid_rows(krows, ctx);
    if (q.D == 128)
      simt_dkdv_kernel<4><<<grid, 256, 0, s>>>(q, k, v, lse, d_o, delta, dk, dv, g, scale, accumulate);
    else
      simt_dkdv_kernel<2><<<grid, 256, 0, s>>>(q, k, v, lse, d_o, delta, dk, dv, g, scale, accumulate);
  }
  timing_end(kKidSimtBwd, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

}  // namespace lsx
