// decode.cu -- split-KV decode partials: one query token per (batch, query
// head) against a long key/value cache cut into chunks; each chunk yields a
// partial (O, LSE) that the one-pass tree merge then reduces (Tree Attention
// abstract: tree reduction across the sequence axis; Lean Attention
// abstract: split the decode over the context and reduce the partials).
//
// Bound: HBM bandwidth.  Every key and value row of the cache is read once
// per key/value head (the G query heads of a group share it), so the
// algorithmic traffic is the cache size.
//
// Decomposition: one CTA of 8 warps per (batch, kv head, chunk).  A warp
// takes 32/G consecutive keys per step (G = query heads per kv head), lane l
// holding elements [4l, 4l+4) of every row, so each row is one coalesced
// 256-byte access.  The G x (32/G) partial dot products are folded with a
// 31-shuffle transpose-reduce that leaves score (key l / G, head l % G) in
// lane l.  Each warp keeps an online softmax per head; the 8 warp states are
// merged in shared memory at the end with the LSE rule.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace lsx {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kWarps = 8;

struct DecodeParams {
  const __nv_bfloat16* q;
  int64_t q_sb, q_sh;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t k_sb, k_sh, k_sn, v_sb, v_sh, v_sn;
  int64_t Hq, Hkv, N, chunk_len, rows;
  float scale_log2;
  float* part_o;
  float* part_l;
};

__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(p));
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  x[0] = __low2float(a); x[1] = __high2float(a);
  x[2] = __low2float(b); x[3] = __high2float(b);
}

template <int G>
__global__ void __launch_bounds__(256) decode_partials_kernel(DecodeParams p) {
  constexpr int KPI = 32 / G;  // keys per warp step
  __shared__ float s_m[kWarps][G];
  __shared__ float s_l[kWarps][G];
  __shared__ float s_o[kWarps][G][128];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t chunk = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int64_t k0 = chunk * p.chunk_len;
  const int64_t k1 = (k0 + p.chunk_len < p.N) ? k0 + p.chunk_len : p.N;

  float qv[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    load4(p.q + b * p.q_sb + (hk * G + g) * p.q_sh + lane * 4, qv[g]);
#pragma unroll
    for (int e = 0; e < 4; ++e) qv[g][e] *= p.scale_log2;
  }
  const __nv_bfloat16* kp = p.k + b * p.k_sb + hk * p.k_sh + lane * 4;
  const __nv_bfloat16* vp = p.v + b * p.v_sb + hk * p.v_sh + lane * 4;

  float m = kNegInf, l = 0.f;  // state of head (lane % G)
  float o[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[g][e] = 0.f;

  for (int64_t base = k0 + warp * KPI; base < k1; base += kWarps * KPI) {
    float kr[KPI][4], vr[KPI][4];
#pragma unroll
    for (int kk = 0; kk < KPI; ++kk) {
      if (base + kk < k1) {
        load4(kp + (base + kk) * p.k_sn, kr[kk]);
        load4(vp + (base + kk) * p.v_sn, vr[kk]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) { kr[kk][e] = 0.f; vr[kk][e] = 0.f; }
      }
    }
    // partial dots, index i = kk * G + g
    float part[32];
#pragma unroll
    for (int kk = 0; kk < KPI; ++kk)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) a = fmaf(qv[g][e], kr[kk][e], a);
        part[kk * G + g] = a;
      }
    // transpose-reduce: afterwards part[0] = full sum of index `lane`
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
      const bool up = (lane & half) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = up ? part[i] : part[i + half];
        const float keep = up ? part[i + half] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
      }
    }
    float s = part[0];
    if (base + lane / G >= k1) s = kNegInf;
    // online softmax for head lane % G over the KPI keys of this step
    float mx = s;
#pragma unroll
    for (int off = G; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m, mx);
    const float alpha = (m == kNegInf) ? 0.f : ex2(m - m_new);
    const float mu = (m_new == kNegInf) ? 0.f : m_new;
    const float pr = ex2(s - mu);
    float ps = pr;
#pragma unroll
    for (int off = G; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
    m = m_new;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float ag = __shfl_sync(0xffffffffu, alpha, g);
#pragma unroll
      for (int e = 0; e < 4; ++e) o[g][e] *= ag;
    }
#pragma unroll
    for (int kk = 0; kk < KPI; ++kk)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pkg = __shfl_sync(0xffffffffu, pr, kk * G + g);
#pragma unroll
        for (int e = 0; e < 4; ++e) o[g][e] = fmaf(pkg, vr[kk][e], o[g][e]);
      }
  }
  // merge the warps' states
  if (lane < G) {
    s_m[warp][lane] = m;
    s_l[warp][lane] = l;
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) s_o[warp][g][lane * 4 + e] = o[g][e];
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * 128; idx += blockDim.x) {
    const int g = idx / 128, d = idx % 128;
    float mm = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, s_m[w][g]);
    float tot = 0.f, acc = 0.f;
    if (mm != kNegInf) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sc = (s_m[w][g] == kNegInf) ? 0.f : ex2(s_m[w][g] - mm);
        tot += s_l[w][g] * sc;
        acc += s_o[w][g][d] * sc;
      }
    }
    const int64_t row = b * p.Hq + hk * G + g;
    p.part_o[(chunk * p.rows + row) * 128 + d] = (tot > 0.f) ? acc / tot : 0.f;
    if (d == 0)
      p.part_l[chunk * p.rows + row] = (tot > 0.f) ? (mm + lg2(tot)) * kLn2 : kNegInf;
  }
}

}  // namespace

int launch_decode_partials(const lsx_tensor& q, const lsx_tensor& kc,
                           const lsx_tensor& vc, int64_t chunk_len,
                           float scale, float* part_o, float* part_lse,
                           const DeviceCtx& ctx, cudaStream_t s) {
  (void)ctx;
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q.data);
  p.q_sb = q.stride_b; p.q_sh = q.stride_h;
  p.k = static_cast<const __nv_bfloat16*>(kc.data);
  p.v = static_cast<const __nv_bfloat16*>(vc.data);
  p.k_sb = kc.stride_b; p.k_sh = kc.stride_h; p.k_sn = kc.stride_n;
  p.v_sb = vc.stride_b; p.v_sh = vc.stride_h; p.v_sn = vc.stride_n;
  p.Hq = q.H; p.Hkv = kc.H; p.N = kc.N; p.chunk_len = chunk_len;
  p.rows = q.B * q.H;
  p.scale_log2 = scale * kLog2e;
  p.part_o = part_o; p.part_l = part_lse;
  const int64_t parts = ceil_div(kc.N, chunk_len);
  if (parts > 65535 * 1024LL || kc.H > 65535 || q.B > 65535) return LSX_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(parts), static_cast<unsigned>(kc.H),
            static_cast<unsigned>(q.B));
  timing_begin(kKidDecode, s);
  switch (q.H / kc.H) {
    case 1: decode_partials_kernel<1><<<grid, 256, 0, s>>>(p); break;
    case 2: decode_partials_kernel<2><<<grid, 256, 0, s>>>(p); break;
    case 4: decode_partials_kernel<4><<<grid, 256, 0, s>>>(p); break;
    case 8: decode_partials_kernel<8><<<grid, 256, 0, s>>>(p); break;
    default: return LSX_ERR_UNSUPPORTED;
  }
  timing_end(kKidDecode, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

}  // namespace lsx
