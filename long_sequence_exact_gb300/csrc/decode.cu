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
// Decomposition: one CTA of 8 compute warps per (batch, kv head, chunk).  A warp
// takes 32/G consecutive keys per step (G = query heads per kv head), lane l
// holding elements [4l, 4l+4) of every row, so each row is one coalesced
// 256-byte access.  The G x (32/G) partial dot products are folded with a
// 31-shuffle transpose-reduce that leaves score (key l / G, head l % G) in
// lane l.  Each warp keeps an online softmax per head; the 8 warp states are
// merged in shared memory at the end with the LSE rule.
//
// Two forms of the same arithmetic:
//  * decode_tma_kernel (G = 2, 4, 8): a ninth warp streams the chunk through a
//    ring of shared-memory stages with TMA (one stage = one key block per
//    compute warp, K and V), so that tens of kilobytes per SM are in flight
//    while the compute warps reduce; the compute warps read rows from shared
//    memory.
//  * decode_partials_kernel (any G, and any layout the TMA maps reject):
//    each warp loads its rows into registers itself.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

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
  int* status;
  uint64_t wait_ns;
  int64_t G;      // query heads per kv head
  int64_t part0;  // first partial block written (chunk c writes part0 + c)
  int64_t qb0;    // query batch of cache batch 0 (row r of a CTA adds r / G)
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
    p.part_o[((p.part0 + chunk) * p.rows + row) * 128 + d] = (tot > 0.f) ? acc / tot : 0.f;
    if (d == 0)
      p.part_l[(p.part0 + chunk) * p.rows + row] = (tot > 0.f) ? (mm + lg2(tot)) * kLn2 : kNegInf;
  }
}

// Rows per CTA, R = GW * RG: every query row that reads this CTA's cache
// chunk (the G heads of a kv head, or, for a shared prefix, the G heads of
// every branch).  Warp w takes rows [GW (w % RG), GW (w % RG) + GW) and key
// group w / RG of KG = 8 / RG; per stage it runs kSub sub-steps of
// KPI = 32 / GW keys, so every (row, key) pair of a stage is scored by one
// warp and each row's partial states come from the KG warps of its group.
template <int GW, int RG>
struct DecodeTmaCfg {
  static constexpr int kR = GW * RG;
  static constexpr int kKpi = 32 / GW;
  static constexpr int kKg = kWarps / RG;
  static constexpr int kSub = (kKg * kKpi >= 64) ? 1 : 64 / (kKg * kKpi);
  static constexpr int kKeys = kKg * kKpi * kSub;   // keys per stage
  static constexpr int kStages = kKeys >= 128 ? 2 : 3;
  static constexpr int kBox = kKeys * 128;          // one [kKeys][64] bf16 box
  static constexpr int kStageBytes = 4 * kBox;      // K and V, two boxes each
  static constexpr int kSmem = kStages * kStageBytes + 256;
};

// Row r, elements [4 lane, 4 lane + 4) of a stage tile stored as two
// [kKeys][64] boxes (columns 0..63, then 64..127).
__device__ __forceinline__ void row4(const uint8_t* tile, int box_bytes, int r, int lane,
                                     float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(tile + (lane >> 4) * box_bytes + r * 128 +
                                                  (lane & 15) * 8);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  x[0] = __low2float(a); x[1] = __high2float(a);
  x[2] = __low2float(b); x[3] = __high2float(b);
}

// Grid (chunks, Hkv, cache batches).  Query row r of a CTA is query head
// hk G + r % G of query batch (cache batch + r / G); its partial goes to
// row (that batch) Hq + head of the partial block `part0 + chunk`.
template <int GW, int RG>
__global__ void __launch_bounds__(32 * (kWarps + 1), GW == 8 ? 1 : 2)
    decode_tma_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, DecodeParams p) {
  using C = DecodeTmaCfg<GW, RG>;
  constexpr int KPI = C::kKpi;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                               ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  int* abort_flag = reinterpret_cast<int*>(empty + C::kStages);
  __shared__ float s_m[kWarps][GW];
  __shared__ float s_l[kWarps][GW];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t chunk = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int64_t k0 = chunk * p.chunk_len;
  const int64_t k1 = (k0 + p.chunk_len < p.N) ? k0 + p.chunk_len : p.N;
  const int64_t n_steps = (k1 - k0 + C::kKeys - 1) / C::kKeys;
  const WaitGuard guard{p.status, p.wait_ns, abort_flag};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int rg = warp % RG, kg = warp / RG;
  float m = kNegInf, l = 0.f;  // state of row GW rg + lane % GW
  float o[GW][4];
#pragma unroll
  for (int g = 0; g < GW; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[g][e] = 0.f;

  if (warp == kWarps) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int64_t s = 0; s < n_steps; ++s) {
        const int stg = static_cast<int>(s % C::kStages);
        const uint32_t round = static_cast<uint32_t>(s / C::kStages);
        if (round > 0 && !mbar_wait(&empty[stg], (round & 1) ^ 1, guard)) break;
        uint8_t* dst = stages + stg * C::kStageBytes;
        const int row = static_cast<int>(k0 + s * C::kKeys);
        mbar_arrive_expect_tx(&full[stg], C::kStageBytes);
        for (int half = 0; half < 2; ++half) {
          tma_load_4d(dst + half * C::kBox, &tm_k, &full[stg], half * 64, row,
                      static_cast<int>(hk), static_cast<int>(b));
          tma_load_4d(dst + (2 + half) * C::kBox, &tm_v, &full[stg], half * 64, row,
                      static_cast<int>(hk), static_cast<int>(b));
        }
      }
    }
  } else {
    // ------------------------------------------------------- compute warps
    float qv[GW][4];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      const int r = rg * GW + g;
      load4(p.q + (p.qb0 + b + r / p.G) * p.q_sb + (hk * p.G + r % p.G) * p.q_sh + lane * 4,
            qv[g]);
#pragma unroll
      for (int e = 0; e < 4; ++e) qv[g][e] *= p.scale_log2;
    }
    for (int64_t s = 0; s < n_steps; ++s) {
      const int stg = static_cast<int>(s % C::kStages);
      if (!mbar_wait(&full[stg], static_cast<uint32_t>(s / C::kStages) & 1, guard)) break;
      const uint8_t* kt = stages + stg * C::kStageBytes;
      const uint8_t* vt = kt + 2 * C::kBox;
      for (int u = 0; u < C::kSub; ++u) {
        const int r0 = (u * C::kKg + kg) * KPI;  // first key of the sub-step in the stage
        const int64_t base = k0 + s * C::kKeys + r0;
        // partial dots, index i = kk * GW + g
        float part[32];
#pragma unroll
        for (int kk = 0; kk < KPI; ++kk) {
          float kr[4];
          row4(kt, C::kBox, r0 + kk, lane, kr);
#pragma unroll
          for (int g = 0; g < GW; ++g) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) a = fmaf(qv[g][e], kr[e], a);
            part[kk * GW + g] = a;
          }
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
        float sc = part[0];
        if (base + lane / GW >= k1) sc = kNegInf;  // past the chunk (zero-filled rows)
        float mx = sc;
#pragma unroll
        for (int off = GW; off < 32; off <<= 1)
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m, mx);
        const float alpha = (m == kNegInf) ? 0.f : ex2(m - m_new);
        const float mu = (m_new == kNegInf) ? 0.f : m_new;
        const float pr = ex2(sc - mu);
        float ps = pr;
#pragma unroll
        for (int off = GW; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l = l * alpha + ps;
        m = m_new;
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          const float ag = __shfl_sync(0xffffffffu, alpha, g);
#pragma unroll
          for (int e = 0; e < 4; ++e) o[g][e] *= ag;
        }
#pragma unroll
        for (int kk = 0; kk < KPI; ++kk) {
          float vr[4];
          row4(vt, C::kBox, r0 + kk, lane, vr);
#pragma unroll
          for (int g = 0; g < GW; ++g) {
            const float pkg = __shfl_sync(0xffffffffu, pr, kk * GW + g);
#pragma unroll
            for (int e = 0; e < 4; ++e) o[g][e] = fmaf(pkg, vr[e], o[g][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stg]);  // this warp is done with the stage
    }
  }
  // merge the warps' states; the per-warp O rows reuse the stage memory once
  // every stage has been consumed
  __syncthreads();
  float* s_o = reinterpret_cast<float*>(stages);  // [kWarps][GW][128]
  if (warp < kWarps) {
    if (lane < GW) {
      s_m[warp][lane] = m;
      s_l[warp][lane] = l;
    }
#pragma unroll
    for (int g = 0; g < GW; ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e) s_o[(warp * GW + g) * 128 + lane * 4 + e] = o[g][e];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < C::kR * 128; idx += blockDim.x) {
    const int r = idx / 128, d = idx % 128;
    const int rgr = r / GW, g = r % GW;
    float mm = kNegInf;
    for (int w = rgr; w < kWarps; w += RG) mm = fmaxf(mm, s_m[w][g]);
    float tot = 0.f, acc = 0.f;
    if (mm != kNegInf) {
      for (int w = rgr; w < kWarps; w += RG) {
        const float f = (s_m[w][g] == kNegInf) ? 0.f : ex2(s_m[w][g] - mm);
        tot += s_l[w][g] * f;
        acc += s_o[(w * GW + g) * 128 + d] * f;
      }
    }
    const int64_t row = (p.qb0 + b + r / p.G) * p.Hq + hk * p.G + r % p.G;
    const int64_t part = p.part0 + chunk;
    p.part_o[(part * p.rows + row) * 128 + d] = (tot > 0.f) ? acc / tot : 0.f;
    if (d == 0)
      p.part_l[part * p.rows + row] = (tot > 0.f) ? (mm + lg2(tot)) * kLn2 : kNegInf;
  }
}

template <int GW, int RG>
bool launch_decode_tma(const lsx_tensor& kc, const lsx_tensor& vc, const DecodeParams& p,
                       dim3 grid, cudaStream_t s) {
  using C = DecodeTmaCfg<GW, RG>;
  CUtensorMap tk, tv;
  if (!make_map_bf16_4d(&tk, kc.data, kc.B, kc.H, kc.N, kc.D, kc.stride_b, kc.stride_h,
                        kc.stride_n, C::kKeys, false) ||
      !make_map_bf16_4d(&tv, vc.data, vc.B, vc.H, vc.N, vc.D, vc.stride_b, vc.stride_h,
                        vc.stride_n, C::kKeys, false))
    return false;  // layout the TMA cannot describe: the register kernel runs
  if (cudaFuncSetAttribute(decode_tma_kernel<GW, RG>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess)
    return false;
  decode_tma_kernel<GW, RG><<<grid, 32 * (kWarps + 1), C::kSmem, s>>>(tk, tv, p);
  return true;
}

// ---------------------------------------------------------------------------
// Tensor-core form for many query rows per cache (a shared prefix read by
// the queries of several branches): R = 16 MT rows, warp w takes the 16-row
// tile w % MT and a 16-key block of every stage (key group w / MT of
// KG = 8 / MT); S = Q K^T and O += P V run as m16n8k16 warp MMAs with
// fragments read by ldmatrix from 128-byte-swizzled TMA stages, P staying in
// registers between the two products.  Per stage: 16 KG keys.
template <int MT>
struct DecodeMmaCfg {
  static constexpr int kR = 16 * MT;
  static constexpr int kKg = kWarps / MT;
  static constexpr int kKeys = 16 * kKg;
  static constexpr int kBox = kKeys * 128;       // one [kKeys][64] bf16 box (swizzled)
  static constexpr int kStageBytes = 4 * kBox;   // K and V, two boxes each
  static constexpr int kStages = kStageBytes >= 65536 ? 2 : (kStageBytes >= 32768 ? 3 : 4);
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
};

// Shared address of the 16-byte chunk c (of 16 per 128-element row) of row r
// in a stage tensor stored as two 128-byte-swizzled [rows][64] boxes.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int box_bytes, int r, int c) {
  return base + (c >> 3) * box_bytes + r * 128 + ((((c & 7) ^ (r & 7))) << 4);
}

template <int MT>
__global__ void __launch_bounds__(32 * (kWarps + 1), 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, DecodeParams p) {
  using C = DecodeMmaCfg<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  int* abort_flag = reinterpret_cast<int*>(empty + C::kStages);
  __shared__ float s_m[kWarps][16];
  __shared__ float s_l[kWarps][16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tid4 = lane & 3;
  const int64_t chunk = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int64_t k0 = chunk * p.chunk_len;
  const int64_t k1 = (k0 + p.chunk_len < p.N) ? k0 + p.chunk_len : p.N;
  const int64_t n_steps = (k1 - k0 + C::kKeys - 1) / C::kKeys;
  const WaitGuard guard{p.status, p.wait_ns, abort_flag};
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int mt = warp % MT, kg = warp / MT;
  float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;  // rows gid, gid + 8
  float o[16][4];
#pragma unroll
  for (int t = 0; t < 16; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[t][e] = 0.f;

  if (warp == kWarps) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int64_t s = 0; s < n_steps; ++s) {
        const int stg = static_cast<int>(s % C::kStages);
        const uint32_t round = static_cast<uint32_t>(s / C::kStages);
        if (round > 0 && !mbar_wait(&empty[stg], (round & 1) ^ 1, guard)) break;
        uint8_t* dst = stages + stg * C::kStageBytes;
        const int row = static_cast<int>(k0 + s * C::kKeys);
        mbar_arrive_expect_tx(&full[stg], C::kStageBytes);
        for (int half = 0; half < 2; ++half) {
          tma_load_4d(dst + half * C::kBox, &tm_k, &full[stg], half * 64, row,
                      static_cast<int>(hk), static_cast<int>(b));
          tma_load_4d(dst + (2 + half) * C::kBox, &tm_v, &full[stg], half * 64, row,
                      static_cast<int>(hk), static_cast<int>(b));
        }
      }
    }
  } else {
    // ------------------------------------------------------- compute warps
    // Q fragments of rows 16 mt + gid (+8), all eight 16-wide K steps of d
    uint32_t qa[8][4];
    {
      const int r0 = 16 * mt + gid, r1 = r0 + 8;
      const __nv_bfloat16* q0 =
          p.q + (p.qb0 + b + r0 / p.G) * p.q_sb + (hk * p.G + r0 % p.G) * p.q_sh;
      const __nv_bfloat16* q1 =
          p.q + (p.qb0 + b + r1 / p.G) * p.q_sb + (hk * p.G + r1 % p.G) * p.q_sh;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int d = 16 * ks + 2 * tid4;
        qa[ks][0] = *reinterpret_cast<const uint32_t*>(q0 + d);
        qa[ks][1] = *reinterpret_cast<const uint32_t*>(q1 + d);
        qa[ks][2] = *reinterpret_cast<const uint32_t*>(q0 + d + 8);
        qa[ks][3] = *reinterpret_cast<const uint32_t*>(q1 + d + 8);
      }
    }
    const float sl2 = p.scale_log2;
    const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix and row of this lane
    for (int64_t s = 0; s < n_steps; ++s) {
      const int stg = static_cast<int>(s % C::kStages);
      if (!mbar_wait(&full[stg], static_cast<uint32_t>(s / C::kStages) & 1, guard)) break;
      const uint32_t kbase = smem_addr(stages + stg * C::kStageBytes);
      const uint32_t vbase = kbase + 2 * C::kBox;
      const int blk = 16 * kg;  // first key of this warp's block in the stage
      // S[16 x 16] = Q K^T: matrices (keys 0-7 | 8-15) x (d chunk 2ks | 2ks+1)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t kb[4];
        ldsm_x4(chunk_addr(kbase, C::kBox, blk + (mi >> 1) * 8 + ri, 2 * ks + (mi & 1)), kb);
        mma_16816(sc[0], qa[ks], kb[0], kb[1]);
        mma_16816(sc[1], qa[ks], kb[2], kb[3]);
      }
      // online softmax of rows gid (elements 0, 1) and gid + 8 (2, 3)
      const int64_t key0 = k0 + s * C::kKeys + blk;
      float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t key = key0 + nt * 8 + 2 * tid4 + (e & 1);
          const float v = key < k1 ? sc[nt][e] * sl2 : kNegInf;
          sc[nt][e] = v;
          if (e < 2) mx_a = fmaxf(mx_a, v); else mx_b = fmaxf(mx_b, v);
        }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float al_a = (m_a == kNegInf) ? 0.f : ex2(m_a - mn_a);
      const float al_b = (m_b == kNegInf) ? 0.f : ex2(m_b - mn_b);
      const float mu_a = (mn_a == kNegInf) ? 0.f : mn_a;
      const float mu_b = (mn_b == kNegInf) ? 0.f : mn_b;
      m_a = mn_a;
      m_b = mn_b;
      float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float pe = ex2(sc[nt][e] - (e < 2 ? mu_a : mu_b));
          sc[nt][e] = pe;
          if (e < 2) ps_a += pe; else ps_b += pe;
        }
      l_a = l_a * al_a + ps_a;
      l_b = l_b * al_b + ps_b;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        o[t][0] *= al_a; o[t][1] *= al_a;
        o[t][2] *= al_b; o[t][3] *= al_b;
      }
      // P as the A fragment of O += P V (k = the 16 keys)
      uint32_t pa[4];
      pa[0] = pack_bf16(sc[0][0], sc[0][1]);
      pa[1] = pack_bf16(sc[0][2], sc[0][3]);
      pa[2] = pack_bf16(sc[1][0], sc[1][1]);
      pa[3] = pack_bf16(sc[1][2], sc[1][3]);
      // V fragments: transposed matrices (keys 0-7 | 8-15) x (d chunk t | t+1)
#pragma unroll
      for (int t2 = 0; t2 < 8; ++t2) {
        uint32_t vb[4];
        ldsm_x4_t(chunk_addr(vbase, C::kBox, blk + (mi & 1) * 8 + ri, 2 * t2 + (mi >> 1)), vb);
        mma_16816(o[2 * t2], pa, vb[0], vb[1]);
        mma_16816(o[2 * t2 + 1], pa, vb[2], vb[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stg]);  // this warp is done with the stage
    }
    // row sums over the four lanes that share a row
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  }
  // merge the KG warps of each 16-row tile; the per-warp O rows reuse the
  // stage memory once every stage has been consumed
  __syncthreads();
  float* s_o = reinterpret_cast<float*>(stages);  // [kWarps][16][128]
  if (warp < kWarps) {
    if (tid4 == 0) {
      s_m[warp][gid] = m_a;
      s_m[warp][gid + 8] = m_b;
      s_l[warp][gid] = l_a;
      s_l[warp][gid + 8] = l_b;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      const int d = 8 * t + 2 * tid4;
      s_o[(warp * 16 + gid) * 128 + d] = o[t][0];
      s_o[(warp * 16 + gid) * 128 + d + 1] = o[t][1];
      s_o[(warp * 16 + gid + 8) * 128 + d] = o[t][2];
      s_o[(warp * 16 + gid + 8) * 128 + d + 1] = o[t][3];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < C::kR * 128; idx += blockDim.x) {
    const int r = idx / 128, d = idx % 128;
    const int tile = r / 16, rr = r % 16;
    float mm = kNegInf;
    for (int w = tile; w < kWarps; w += MT) mm = fmaxf(mm, s_m[w][rr]);
    float tot = 0.f, acc = 0.f;
    if (mm != kNegInf) {
      for (int w = tile; w < kWarps; w += MT) {
        const float f = (s_m[w][rr] == kNegInf) ? 0.f : ex2(s_m[w][rr] - mm);
        tot += s_l[w][rr] * f;
        acc += s_o[(w * 16 + rr) * 128 + d] * f;
      }
    }
    const int64_t row = (p.qb0 + b + r / p.G) * p.Hq + hk * p.G + r % p.G;
    const int64_t part = p.part0 + chunk;
    p.part_o[(part * p.rows + row) * 128 + d] = (tot > 0.f) ? acc / tot : 0.f;
    if (d == 0)
      p.part_l[part * p.rows + row] = (tot > 0.f) ? (mm + lg2(tot)) * kLn2 : kNegInf;
  }
}

template <int MT>
bool launch_decode_mma(const lsx_tensor& kc, const lsx_tensor& vc, const DecodeParams& p,
                       dim3 grid, cudaStream_t s) {
  using C = DecodeMmaCfg<MT>;
  CUtensorMap tk, tv;
  if (!make_map_bf16_4d(&tk, kc.data, kc.B, kc.H, kc.N, kc.D, kc.stride_b, kc.stride_h,
                        kc.stride_n, C::kKeys) ||
      !make_map_bf16_4d(&tv, vc.data, vc.B, vc.H, vc.N, vc.D, vc.stride_b, vc.stride_h,
                        vc.stride_n, C::kKeys))
    return false;
  if (cudaFuncSetAttribute(decode_mma_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmem) != cudaSuccess)
    return false;
  decode_mma_kernel<MT><<<grid, 32 * (kWarps + 1), C::kSmem, s>>>(tk, tv, p);
  return true;
}

// Rows per CTA R (a multiple of 2 up to 64): picks the (GW, RG) instance.
// Sixteen rows or more take the tensor-core form.
bool launch_decode_rows(int64_t R, const lsx_tensor& kc, const lsx_tensor& vc,
                        const DecodeParams& p, dim3 grid, cudaStream_t s) {
  switch (R) {
    case 16: return launch_decode_mma<1>(kc, vc, p, grid, s);
    case 32: return launch_decode_mma<2>(kc, vc, p, grid, s);
    case 64: return launch_decode_mma<4>(kc, vc, p, grid, s);
    default: break;
  }
  switch (R) {
    case 2: return launch_decode_tma<2, 1>(kc, vc, p, grid, s);
    case 4: return launch_decode_tma<4, 1>(kc, vc, p, grid, s);
    case 8: return launch_decode_tma<8, 1>(kc, vc, p, grid, s);
    case 16: return launch_decode_tma<8, 2>(kc, vc, p, grid, s);
    case 32: return launch_decode_tma<8, 4>(kc, vc, p, grid, s);
    case 64: return launch_decode_tma<8, 8>(kc, vc, p, grid, s);
    default: return false;
  }
}

}  // namespace

namespace {
DecodeParams decode_params(const lsx_tensor& q, const lsx_tensor& kc, const lsx_tensor& vc,
                           int64_t chunk_len, float scale, float* part_o, float* part_lse,
                           int64_t part0, const DeviceCtx& ctx) {
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
  p.status = ctx.status; p.wait_ns = ctx.wait_ns;
  p.G = q.H / kc.H;
  p.part0 = part0;
  p.qb0 = 0;
  return p;
}
}  // namespace

int launch_decode_partials(const lsx_tensor& q, const lsx_tensor& kc,
                           const lsx_tensor& vc, int64_t chunk_len,
                           float scale, float* part_o, float* part_lse,
                           const DeviceCtx& ctx, cudaStream_t s, int64_t part0) {
  DecodeParams p = decode_params(q, kc, vc, chunk_len, scale, part_o, part_lse, part0, ctx);
  const int64_t parts = ceil_div(kc.N, chunk_len);
  if (parts > 65535 * 1024LL || kc.H > 65535 || q.B > 65535) return LSX_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(parts), static_cast<unsigned>(kc.H),
            static_cast<unsigned>(q.B));
  timing_begin(kKidDecode, s);
  bool done = p.G >= 2 && launch_decode_rows(p.G, kc, vc, p, grid, s);
  if (!done) switch (q.H / kc.H) {
    case 1: decode_partials_kernel<1><<<grid, 256, 0, s>>>(p); break;
    case 2: decode_partials_kernel<2><<<grid, 256, 0, s>>>(p); break;
    case 4: decode_partials_kernel<4><<<grid, 256, 0, s>>>(p); break;
    case 8: decode_partials_kernel<8><<<grid, 256, 0, s>>>(p); break;
    default: return LSX_ERR_UNSUPPORTED;
  }
  timing_end(kKidDecode, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

// Partials of every branch's queries against one shared cache (batch 1):
// the branches are taken `group` at a time, each group's B_g * G query rows
// reading the cache once (DeFT, KV-guided grouping).
int launch_decode_shared(const lsx_tensor& q, const lsx_tensor& kc, const lsx_tensor& vc,
                         int64_t chunk_len, float scale, float* part_o, float* part_lse,
                         const DeviceCtx& ctx, cudaStream_t s, int64_t part0) {
  DecodeParams p = decode_params(q, kc, vc, chunk_len, scale, part_o, part_lse, part0, ctx);
  const int64_t parts = ceil_div(kc.N, chunk_len);
  if (parts > 65535 * 1024LL || kc.H > 65535) return LSX_ERR_UNSUPPORTED;
  if (q.B == 1)  // one branch: the cache's batch is the query's
    return launch_decode_partials(q, kc, vc, chunk_len, scale, part_o, part_lse, ctx, s, part0);
  // largest power-of-two branch group with group * G rows <= 64
  int64_t group = 1;
  while (group * 2 <= q.B && group * 2 * p.G <= 64) group *= 2;
  dim3 grid(static_cast<unsigned>(parts), static_cast<unsigned>(kc.H), 1u);
  timing_begin(kKidDecode, s);
  for (int64_t b0 = 0; b0 < q.B;) {
    int64_t g = group;
    while (g > q.B - b0) g /= 2;  // the tail: the largest power of two that fits
    int64_t start = b0;
    if (g * p.G < 2) {  // one query row left (G = 1): redo the last two branches
      g = 2;
      start = q.B - 2;
    }
    p.qb0 = start;
    if (!launch_decode_rows(g * p.G, kc, vc, p, grid, s)) {
      timing_end(kKidDecode, s);
      return LSX_ERR_UNSUPPORTED;
    }
    b0 = start + g;
  }
  timing_end(kKidDecode, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

}  // namespace lsx
