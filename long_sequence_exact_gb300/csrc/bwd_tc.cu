// bwd_tc.cu -- tcgen05 backward of exact attention over a chunk pair, from
// the SAVED final output and log-sum-exp (DistFlashAttn, core concepts:
// rematerialization-aware checkpointing -- the forward pass is not re-run;
// only the score tiles are rebuilt from Q, K and the saved LSE).
//
// With P_ij = exp(scale <q_i,k_j> - LSE_i), delta_i = <dO_i, O_i> (computed
// beforehand by the row-dot kernel from the saved O) and
// dS_ij = P_ij (dO_i.v_j - delta_i):
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
//
// Two persistent kernels, both deterministic (every output tile is owned by
// exactly one CTA; no atomics):
//  * dkdv_kernel, key-tile-major: a work item is one 128-row key/value tile
//    of one (batch, kv head); it walks every query tile (of every query head
//    of the group) that sees it:
//      S^T  = K Q_i^T     (SS, K-major x K-major)      TMEM [0,128)
//      dP^T = V dO_i^T    (SS)                         TMEM [128,256)
//      grad warps: P^T, dS^T -> bf16 back into TMEM (inside [0,128), [128,256))
//      dV  += P^T dO_i    (TS, dO_i MN-major)          TMEM [256,256+D)
//      dK  += dS^T Q_i    (TS, Q_i MN-major)           TMEM [384,384+D)
//  * dq_kernel, query-tile-major: a work item is one 128-row query tile; it
//    walks every visible key tile:
//      S  = Q K_j^T, dP = dO V_j^T (SS)                TMEM [0,128), [128,256)
//      grad warps: dS -> bf16 into TMEM (inside [128,256))
//      dQ += dS K_j       (TS, K_j MN-major)           TMEM [256,256+D)
// Roles per CTA (384 threads): warp 0 loads (TMA), warp 1 owns TMEM and
// issues the MMAs (lane 0), warps 4..11 compute P and dS and write the
// outputs.  Grad warp g covers TMEM lanes 32 (g % 4) .. +31 and the half
// g / 4 of the 128 columns; each half packs its bf16 result into the first
// 32 columns of its own 64, so the two warps sharing a lane range never
// touch each other's columns, and the TS MMAs address each 16-wide K step
// of the bf16 operand at packed_col(kk).
// MMA issue order: the next step's S/dP products are issued right after the
// current dV/dK (dQ) products without waiting for them; one thread's
// tcgen05.mma operations execute in issue order, so the bf16 operands read
// by the earlier MMAs are consumed before the later MMAs overwrite them.
// Work items are dealt longest-first in snake order.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace lsx {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int64_t B, Hq, Hkv, Lq, Lk;
  int64_t q_off, kv_off;
  int causal, accumulate;
  float scale_log2;  // scale * log2(e)
  float scale;
  const float* lse;
  int64_t l_sb, l_sh, l_sn;
  const float* delta;  // dense [B*Hq*Lq]
  void* dq;
  int dq_f32;
  int64_t dq_sb, dq_sh, dq_sn;
  void* dk;
  int dk_f32;
  int64_t dk_sb, dk_sh, dk_sn;
  void* dv;
  int dv_f32;
  int64_t dv_sb, dv_sh, dv_sn;
  int64_t n_qtiles, n_ktiles;
  int64_t n_items;
  int* status;
  uint64_t wait_ns;
};

// TMEM column (relative to the 128-column fp32 tile) of the packed bf16
// operand for K step kk (16 elements = 8 packed columns).
__device__ __forceinline__ uint32_t packed_col(int kk) {
  return kk < 4 ? static_cast<uint32_t>(kk * 8) : static_cast<uint32_t>(64 + (kk - 4) * 8);
}

// First query tile that sees key tile j (n_qtiles when none does).
__device__ __forceinline__ int64_t q_tile_begin(const BwdParams& p, int64_t j) {
  if (!p.causal) return 0;
  const int64_t need = p.kv_off + 128 * j - p.q_off;  // first query row seeing key 128 j
  if (need <= 0) return 0;
  if (need > p.Lq - 1) return p.n_qtiles;
  return need / 128;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) break;
  }
}

// 32 fp32 values scaled by `mult` and written to a bf16 or f32 output row,
// optionally added to what is there.
__device__ __forceinline__ void store_row32(void* out, int f32, int64_t off,
                                            const uint32_t (&u)[32], float mult,
                                            int accumulate) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]) * mult;
  if (f32) {
    float* dst = static_cast<float*>(out) + off;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float4 w = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      if (accumulate) {
        const float4 o = *reinterpret_cast<const float4*>(dst + i);
        w.x += o.x; w.y += o.y; w.z += o.z; w.w += o.w;
      }
      *reinterpret_cast<float4*>(dst + i) = w;
    }
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + off;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = v[i + e];
      if (accumulate) {
        const uint4 o = *reinterpret_cast<const uint4*>(dst + i);
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&ow[e]);
          x[2 * e] += __low2float(pr);
          x[2 * e + 1] += __high2float(pr);
        }
      }
      uint4 w;
      w.x = pack_bf16(x[0], x[1]);
      w.y = pack_bf16(x[2], x[3]);
      w.z = pack_bf16(x[4], x[5]);
      w.w = pack_bf16(x[6], x[7]);
      *reinterpret_cast<uint4*>(dst + i) = w;
    }
  }
}

// Loads 64 fp32 columns (two x32 loads) of two TMEM tiles with one wait.
__device__ __forceinline__ void ld_two_halves(uint32_t ta, uint32_t tb, uint32_t (&a0)[32],
                                              uint32_t (&a1)[32], uint32_t (&b0)[32],
                                              uint32_t (&b1)[32]) {
  tmem_ld32(ta, a0);
  tmem_ld32(ta + 32, a1);
  tmem_ld32(tb, b0);
  tmem_ld32(tb + 32, b1);
  tmem_ld_wait32(a0);
  reg_fence32(a1);
  reg_fence32(b0);
  reg_fence32(b1);
}

// ===================================================================== dK dV
template <int D>
struct DkdvSmem {
  static constexpr int kStages = 2;
  __nv_bfloat16 k[128 * D];
  __nv_bfloat16 v[128 * D];
  __nv_bfloat16 q[kStages][128 * D];
  __nv_bfloat16 d_o[kStages][128 * D];
  float lse2[kStages][128];   // LSE * log2(e); +inf for rows without keys
  float delta[kStages][128];
  uint64_t kv_full, kv_empty, final_bar;
  uint64_t st_full[kStages], st_empty[kStages];
  uint64_t s_full, p_full, dkv_done;
  uint32_t tmem_base;
  int abort;
};

struct DkdvItem {
  int64_t b, hk, j, i0, n_i, group;
};

__device__ __forceinline__ DkdvItem dkdv_item(const BwdParams& p, int64_t it) {
  DkdvItem x;
  const int64_t bh_n = p.B * p.Hkv;
  x.j = it / bh_n;  // key tile 0 (the most query tiles) first
  const int64_t bh = it % bh_n;
  x.b = bh / p.Hkv;
  x.hk = bh % p.Hkv;
  x.group = p.Hq / p.Hkv;
  x.i0 = q_tile_begin(p, x.j);
  x.n_i = (p.n_qtiles - x.i0) * x.group;  // (head, query tile) steps
  return x;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using Sm = DkdvSmem<D>;
  constexpr int kStages = Sm::kStages;
  constexpr int kTile = 128 * D * 2;
  constexpr int kSub = D / 64;
  extern __shared__ uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                  ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitGuard guard{p.status, p.wait_ns, &sm.abort};
  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    mbar_init(&sm.final_bar, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.st_full[s], 32);
      mbar_init(&sm.st_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, 256);
    mbar_init(&sm.dkv_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int64_t G = gridDim.x, c = blockIdx.x;

  // 384 threads launched at <= 168 registers (64,512): the load/MMA
  // warpgroup keeps 88, the two grad warpgroups take 184:
  // 128 * 88 + 256 * 184 = 58,368 <= 64,512.
  if (warp < 4) {
    regs_dec<88>();
    if (warp == 0) {
      // -------------------------------------------------- loads (warp 0)
      uint32_t stage = 0, phase = 0, kv_phase = 0;
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        const DkdvItem x = dkdv_item(p, it);
        if (!mbar_wait(&sm.kv_empty, kv_phase ^ 1, guard)) break;
        kv_phase ^= 1;
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.kv_full, 2 * kTile);
          for (int sub = 0; sub < kSub; ++sub) {
            tma_load_4d(&sm.k[sub * 128 * 64], &tm_k, &sm.kv_full, sub * 64,
                        static_cast<int>(x.j * 128), static_cast<int>(x.hk),
                        static_cast<int>(x.b));
            tma_load_4d(&sm.v[sub * 128 * 64], &tm_v, &sm.kv_full, sub * 64,
                        static_cast<int>(x.j * 128), static_cast<int>(x.hk),
                        static_cast<int>(x.b));
          }
        }
        bool ok = true;
        for (int64_t s = 0; s < x.n_i; ++s) {
          const int64_t h = x.hk * x.group + s / (p.n_qtiles - x.i0);
          const int64_t i = x.i0 + s % (p.n_qtiles - x.i0);
          if (!mbar_wait(&sm.st_empty[stage], phase ^ 1, guard)) { ok = false; break; }
          // LSE (as log2 units) and delta of the 128 query rows of tile i
          for (int t = lane; t < 128; t += 32) {
            const int64_t row = i * 128 + t;
            float l2 = kPosInf, dl = 0.f;
            if (row < p.Lq) {
              const float lse = p.lse[x.b * p.l_sb + h * p.l_sh + row * p.l_sn];
              l2 = (lse == kNegInf) ? kPosInf : lse * kLog2e;
              dl = p.delta[(x.b * p.Hq + h) * p.Lq + row];
            }
            sm.lse2[stage][t] = l2;
            sm.delta[stage][t] = dl;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&sm.st_full[stage], 2 * kTile);
            for (int sub = 0; sub < kSub; ++sub) {
              tma_load_4d(&sm.q[stage][sub * 128 * 64], &tm_q, &sm.st_full[stage], sub * 64,
                          static_cast<int>(i * 128), static_cast<int>(h), static_cast<int>(x.b));
              tma_load_4d(&sm.d_o[stage][sub * 128 * 64], &tm_do, &sm.st_full[stage],
                          sub * 64, static_cast<int>(i * 128), static_cast<int>(h),
                          static_cast<int>(x.b));
            }
          } else {
            mbar_arrive(&sm.st_full[stage]);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    } else if (warp == 1 && lane == 0) {
      // ----------------------------------------------------------- MMA issue
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, 1);
      uint32_t stage = 0, phase = 0, kv_phase = 0, p_phase = 0;
      bool issued = false;
      const uint32_t k_addr = smem_addr(sm.k), v_addr = smem_addr(sm.v);
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        const DkdvItem x = dkdv_item(p, it);
        if (!mbar_wait(&sm.kv_full, kv_phase, guard)) break;
        kv_phase ^= 1;
        tc_fence_after();
        bool ok = true;
        for (int64_t s = 0; s < x.n_i; ++s) {
          if (!mbar_wait(&sm.st_full[stage], phase, guard)) { ok = false; break; }
          tc_fence_after();
          const uint32_t q_addr = smem_addr(sm.q[stage]);
          const uint32_t o_addr = smem_addr(sm.d_o[stage]);
#pragma unroll 1
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            mma_ss(tmem + 0, sdesc_sw128(k_addr + off, 16, 1024),
                   sdesc_sw128(q_addr + off, 16, 1024), kIdS, kk > 0);
          }
#pragma unroll 1
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            mma_ss(tmem + 128, sdesc_sw128(v_addr + off, 16, 1024),
                   sdesc_sw128(o_addr + off, 16, 1024), kIdS, kk > 0);
          }
          mma_commit(&sm.s_full);
          issued = true;
          if (!mbar_wait(&sm.p_full, p_phase, guard)) { ok = false; break; }
          p_phase ^= 1;
          tc_fence_after();
#pragma unroll 1
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
            mma_ts(tmem + 256, tmem + packed_col(kk),
                   sdesc_sw128(o_addr + kk * 2048, 128 * 128, 1024), kIdG, acc);
            mma_ts(tmem + 384, tmem + 128 + packed_col(kk),
                   sdesc_sw128(q_addr + kk * 2048, 128 * 128, 1024), kIdG, acc);
          }
          mma_commit(&sm.dkv_done);
          mma_commit(&sm.st_empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(&sm.kv_empty);
      }
      if (issued) {
        mma_commit(&sm.final_bar);
        drain_wait(&sm.final_bar, 0, p.wait_ns);
      }
    }
  } else {
    regs_inc<184>();
    // -------------------------------------------- P^T, dS^T and the epilogue
    const int g = warp - 4;
    const int quad = g & 3, half = g >> 2;
    const int row = quad * 32 + lane;  // key row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + 64 * half;        // S^T / P^T
    const uint32_t tP = tmem + lane_base + 128 + 64 * half;  // dP^T / dS^T
    uint32_t stage = 0, phase = 0, s_phase = 0;
    uint32_t d_count = 0;
    const float sl2 = p.scale_log2;
    const float2 sc2 = make_float2(sl2, sl2);
    for (int64_t r = 0;; ++r) {
      const int64_t it = snake_item(c, r, G);
      if (it >= p.n_items) break;
      const DkdvItem x = dkdv_item(p, it);
      const int64_t key_abs = p.kv_off + x.j * 128 + row;
      bool ok = true;
      for (int64_t s = 0; s < x.n_i; ++s) {
        const int64_t i = x.i0 + s % (p.n_qtiles - x.i0);
        if (!mbar_wait(&sm.s_full, s_phase, guard)) { ok = false; break; }
        s_phase ^= 1;
        // the stage's LSE/delta rows were published with st_full
        if (!mbar_wait(&sm.st_full[stage], phase, guard)) { ok = false; break; }
        tc_fence_after();
        uint32_t us0[32], us1[32], ud0[32], ud1[32];
        ld_two_halves(tS, tP, us0, us1, ud0, ud1);
        // query columns c (of this half) with q_off + 128 i + 64 half + c >=
        // key_abs are visible
        int cmin = 0;
        if (p.causal) {
          const int64_t tt = key_abs - (p.q_off + i * 128 + 64 * half);
          cmin = tt <= 0 ? 0 : (tt > 64 ? 64 : static_cast<int>(tt));
        }
        const float4* l2v = reinterpret_cast<const float4*>(&sm.lse2[stage][64 * half]);
        const float4* dlv = reinterpret_cast<const float4*>(&sm.delta[stage][64 * half]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint32_t(&us)[32] = cc ? us1 : us0;
          const uint32_t(&ud)[32] = cc ? ud1 : ud0;
          uint32_t pk[16], dk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 l4 = l2v[cc * 8 + e4];
            const float4 d4 = dlv[cc * 8 + e4];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int e = e4 * 2 + hh;  // pair index within the chunk
              const int c0 = cc * 32 + 2 * e;
              const float2 nl = hh ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
              const float2 nd = hh ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
              const float2 arg = __ffma2_rn(
                  make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sc2, nl);
              float2 pr = make_float2(ex2(arg.x), ex2(arg.y));
              if (c0 < cmin) pr.x = 0.f;
              if (c0 + 1 < cmin) pr.y = 0.f;
              const float2 dpm = __fadd2_rn(
                  make_float2(__uint_as_float(ud[2 * e]), __uint_as_float(ud[2 * e + 1])), nd);
              const float2 ds = __fmul2_rn(pr, dpm);
              pk[e] = pack_bf16(pr.x, pr.y);
              dk[e] = pack_bf16(ds.x, ds.y);
            }
          }
          tmem_st16(tS + cc * 16, pk);
          tmem_st16(tP + cc * 16, dk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full);
        ++d_count;
        if (++stage == DkdvSmem<D>::kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      // epilogue: half 0 writes dV, half 1 writes dK (times scale)
      if (x.n_i > 0) {
        if (!mbar_wait(&sm.dkv_done, (d_count - 1) & 1, guard)) break;
        tc_fence_after();
      }
      const int64_t krow = x.j * 128 + row;
      const bool valid = krow < p.Lk;
      const uint32_t base_col = half == 0 ? 256u : 384u;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t u[32];
        if (x.n_i > 0) {
          tmem_ld32(tmem + lane_base + base_col + cc * 32, u);
          tmem_ld_wait32(u);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        if (!valid) continue;
        if (half == 0)
          store_row32(p.dv, p.dv_f32, x.b * p.dv_sb + x.hk * p.dv_sh + krow * p.dv_sn + cc * 32,
                      u, 1.f, p.accumulate);
        else
          store_row32(p.dk, p.dk_f32, x.b * p.dk_sb + x.hk * p.dk_sh + krow * p.dk_sn + cc * 32,
                      u, p.scale, p.accumulate);
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================= dQ
template <int D>
struct DqSmem {
  static constexpr int kStages = 2;
  __nv_bfloat16 q[128 * D];
  __nv_bfloat16 d_o[128 * D];
  __nv_bfloat16 k[kStages][128 * D];
  __nv_bfloat16 v[kStages][128 * D];
  uint64_t qo_full, qo_empty, final_bar;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full, p_full, dq_done;
  uint32_t tmem_base;
  int abort;
};

struct DqItem {
  int64_t b, h, hk, i, nkv;
};

__device__ __forceinline__ DqItem dq_item(const BwdParams& p, int64_t it) {
  DqItem x;
  const int64_t bh_n = p.B * p.Hq;
  x.i = p.n_qtiles - 1 - it / bh_n;  // the longest key range first
  const int64_t bh = it % bh_n;
  x.b = bh / p.Hq;
  x.h = bh % p.Hq;
  x.hk = x.h / (p.Hq / p.Hkv);
  x.nkv = fwd_kv_tiles(x.i, p.Lq, p.Lk, p.q_off, p.kv_off, p.causal);
  return x;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using Sm = DqSmem<D>;
  constexpr int kStages = Sm::kStages;
  constexpr int kTile = 128 * D * 2;
  constexpr int kSub = D / 64;
  extern __shared__ uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                  ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitGuard guard{p.status, p.wait_ns, &sm.abort};
  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.qo_full, 1);
    mbar_init(&sm.qo_empty, 1);
    mbar_init(&sm.final_bar, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, 256);
    mbar_init(&sm.dq_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int64_t G = gridDim.x, c = blockIdx.x;

  // same register split as dkdv_kernel: 128 * 88 + 256 * 184 <= 384 * 168
  if (warp < 4) {
    regs_dec<88>();
    if (warp == 0 && lane == 0) {
      uint32_t stage = 0, phase = 0, qo_phase = 0;
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        const DqItem x = dq_item(p, it);
        if (!mbar_wait(&sm.qo_empty, qo_phase ^ 1, guard)) break;
        qo_phase ^= 1;
        mbar_arrive_expect_tx(&sm.qo_full, 2 * kTile);
        for (int sub = 0; sub < kSub; ++sub) {
          tma_load_4d(&sm.q[sub * 128 * 64], &tm_q, &sm.qo_full, sub * 64,
                      static_cast<int>(x.i * 128), static_cast<int>(x.h), static_cast<int>(x.b));
          tma_load_4d(&sm.d_o[sub * 128 * 64], &tm_do, &sm.qo_full, sub * 64,
                      static_cast<int>(x.i * 128), static_cast<int>(x.h), static_cast<int>(x.b));
        }
        bool ok = true;
        for (int64_t j = 0; j < x.nkv; ++j) {
          if (!mbar_wait(&sm.kv_empty[stage], phase ^ 1, guard)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.kv_full[stage], 2 * kTile);
          for (int sub = 0; sub < kSub; ++sub) {
            tma_load_4d(&sm.k[stage][sub * 128 * 64], &tm_k, &sm.kv_full[stage], sub * 64,
                        static_cast<int>(j * 128), static_cast<int>(x.hk), static_cast<int>(x.b));
            tma_load_4d(&sm.v[stage][sub * 128 * 64], &tm_v, &sm.kv_full[stage], sub * 64,
                        static_cast<int>(j * 128), static_cast<int>(x.hk), static_cast<int>(x.b));
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    } else if (warp == 1 && lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, 1);
      uint32_t stage = 0, phase = 0, qo_phase = 0, p_phase = 0;
      bool issued = false;
      const uint32_t q_addr = smem_addr(sm.q), o_addr = smem_addr(sm.d_o);
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        const DqItem x = dq_item(p, it);
        if (!mbar_wait(&sm.qo_full, qo_phase, guard)) break;
        qo_phase ^= 1;
        tc_fence_after();
        bool ok = true;
        for (int64_t j = 0; j < x.nkv; ++j) {
          if (!mbar_wait(&sm.kv_full[stage], phase, guard)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_addr = smem_addr(sm.k[stage]);
          const uint32_t v_addr = smem_addr(sm.v[stage]);
#pragma unroll 1
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            mma_ss(tmem + 0, sdesc_sw128(q_addr + off, 16, 1024),
                   sdesc_sw128(k_addr + off, 16, 1024), kIdS, kk > 0);
          }
#pragma unroll 1
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * (128 * 128) + (kk % 4) * 32;
            mma_ss(tmem + 128, sdesc_sw128(o_addr + off, 16, 1024),
                   sdesc_sw128(v_addr + off, 16, 1024), kIdS, kk > 0);
          }
          mma_commit(&sm.s_full);
          issued = true;
          if (!mbar_wait(&sm.p_full, p_phase, guard)) { ok = false; break; }
          p_phase ^= 1;
          tc_fence_after();
#pragma unroll 1
          for (int kk = 0; kk < 8; ++kk) {
            mma_ts(tmem + 256, tmem + 128 + packed_col(kk),
                   sdesc_sw128(k_addr + kk * 2048, 128 * 128, 1024), kIdG,
                   (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&sm.dq_done);
          mma_commit(&sm.kv_empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        mma_commit(&sm.qo_empty);
      }
      if (issued) {
        mma_commit(&sm.final_bar);
        drain_wait(&sm.final_bar, 0, p.wait_ns);
      }
    }
  } else {
    regs_inc<184>();
    const int g = warp - 4;
    const int quad = g & 3, half = g >> 2;
    const int row = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + 64 * half;
    const uint32_t tP = tmem + lane_base + 128 + 64 * half;
    uint32_t s_phase = 0, d_count = 0;
    const float sl2 = p.scale_log2;
    const float2 sc2 = make_float2(sl2, sl2);
    for (int64_t r = 0;; ++r) {
      const int64_t it = snake_item(c, r, G);
      if (it >= p.n_items) break;
      const DqItem x = dq_item(p, it);
      const int64_t qrow = x.i * 128 + row;
      const bool valid = qrow < p.Lq;
      float l2 = kPosInf, dl = 0.f;
      if (valid) {
        const float lse = p.lse[x.b * p.l_sb + x.h * p.l_sh + qrow * p.l_sn];
        l2 = (lse == kNegInf) ? kPosInf : lse * kLog2e;
        dl = p.delta[(x.b * p.Hq + x.h) * p.Lq + qrow];
      }
      const float2 nl = make_float2(-l2, -l2);
      const float2 nd = make_float2(-dl, -dl);
      bool ok = true;
      for (int64_t j = 0; j < x.nkv; ++j) {
        if (!mbar_wait(&sm.s_full, s_phase, guard)) { ok = false; break; }
        s_phase ^= 1;
        tc_fence_after();
        uint32_t us0[32], us1[32], ud0[32], ud1[32];
        ld_two_halves(tS, tP, us0, us1, ud0, ud1);
        // visible key columns of this half: c <= climit
        const int64_t kb = j * 128 + 64 * half;
        int64_t lim = 63;
        if (kb + 64 > p.Lk) lim = p.Lk - kb - 1;
        if (p.causal) {
          const int64_t c2 = p.q_off + qrow - p.kv_off - kb;
          if (c2 < lim) lim = c2;
        }
        const int climit = lim < -1 ? -1 : static_cast<int>(lim);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint32_t(&us)[32] = cc ? us1 : us0;
          const uint32_t(&ud)[32] = cc ? ud1 : ud0;
          uint32_t dk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = cc * 32 + 2 * e;
            const float2 arg = __ffma2_rn(
                make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sc2, nl);
            float2 pr = make_float2(ex2(arg.x), ex2(arg.y));
            if (c0 > climit) pr.x = 0.f;
            if (c0 + 1 > climit) pr.y = 0.f;
            const float2 dpm = __fadd2_rn(
                make_float2(__uint_as_float(ud[2 * e]), __uint_as_float(ud[2 * e + 1])), nd);
            const float2 ds = __fmul2_rn(pr, dpm);
            dk[e] = pack_bf16(ds.x, ds.y);
          }
          tmem_st16(tP + cc * 16, dk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full);
        ++d_count;
      }
      if (!ok) break;
      if (x.nkv > 0) {
        if (!mbar_wait(&sm.dq_done, (d_count - 1) & 1, guard)) break;
        tc_fence_after();
      }
      // epilogue: half h writes dQ columns [D/2 h, D/2 h + D/2) (times scale)
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int col = (D / 2) * half + cc * 32;
        uint32_t u[32];
        if (x.nkv > 0) {
          tmem_ld32(tmem + lane_base + 256 + col, u);
          tmem_ld_wait32(u);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        if (!valid) continue;
        store_row32(p.dq, p.dq_f32, x.b * p.dq_sb + x.h * p.dq_sh + qrow * p.dq_sn + col, u,
                    p.scale, p.accumulate);
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
int launch_bwd_tc_d(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                    const lsx_tensor& lse, const lsx_tensor& d_o, const float* delta,
                    int64_t q_off, int64_t kv_off, int causal, float scale,
                    const lsx_tensor& dq, const lsx_tensor& dk, const lsx_tensor& dv,
                    int accumulate, const DeviceCtx& ctx, cudaStream_t s) {
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map_bf16_4d(&tq, q.data, q.B, q.H, q.N, q.D, q.stride_b, q.stride_h, q.stride_n, 128) ||
      !make_map_bf16_4d(&tk, k.data, k.B, k.H, k.N, k.D, k.stride_b, k.stride_h, k.stride_n, 128) ||
      !make_map_bf16_4d(&tv, v.data, v.B, v.H, v.N, v.D, v.stride_b, v.stride_h, v.stride_n, 128) ||
      !make_map_bf16_4d(&tdo, d_o.data, d_o.B, d_o.H, d_o.N, d_o.D, d_o.stride_b, d_o.stride_h,
                        d_o.stride_n, 128))
    return LSX_ERR_LAUNCH;
  BwdParams p;
  p.B = q.B; p.Hq = q.H; p.Hkv = k.H; p.Lq = q.N; p.Lk = k.N;
  p.q_off = q_off; p.kv_off = kv_off; p.causal = causal; p.accumulate = accumulate;
  p.scale_log2 = scale * kLog2e; p.scale = scale;
  p.lse = static_cast<const float*>(lse.data);
  p.l_sb = lse.stride_b; p.l_sh = lse.stride_h; p.l_sn = lse.stride_n;
  p.delta = delta;
  p.dq = dq.data; p.dq_f32 = dq.dtype == LSX_F32;
  p.dq_sb = dq.stride_b; p.dq_sh = dq.stride_h; p.dq_sn = dq.stride_n;
  p.dk = dk.data; p.dk_f32 = dk.dtype == LSX_F32;
  p.dk_sb = dk.stride_b; p.dk_sh = dk.stride_h; p.dk_sn = dk.stride_n;
  p.dv = dv.data; p.dv_f32 = dv.dtype == LSX_F32;
  p.dv_sb = dv.stride_b; p.dv_sh = dv.stride_h; p.dv_sn = dv.stride_n;
  p.n_qtiles = ceil_div(q.N, 128);
  p.n_ktiles = ceil_div(k.N, 128);
  p.status = ctx.status; p.wait_ns = ctx.wait_ns;

  // dK, dV: items (key tile, b, kv head)
  p.n_items = p.n_ktiles * q.B * k.H;
  {
    const size_t smem = sizeof(DkdvSmem<D>) + 1024;
    if (cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LSX_ERR_LAUNCH;
    const int64_t grid = p.n_items < ctx.sm_count ? p.n_items : ctx.sm_count;
    timing_begin(kKidDkdv, s);
    dkdv_kernel<D><<<static_cast<unsigned>(grid), 384, smem, s>>>(tq, tk, tv, tdo, p);
    timing_end(kKidDkdv, s);
    if (cudaGetLastError() != cudaSuccess) return LSX_ERR_LAUNCH;
  }
  // dQ: items (query tile, b, head)
  p.n_items = p.n_qtiles * q.B * q.H;
  {
    const size_t smem = sizeof(DqSmem<D>) + 1024;
    if (cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LSX_ERR_LAUNCH;
    const int64_t grid = p.n_items < ctx.sm_count ? p.n_items : ctx.sm_count;
    timing_begin(kKidDq, s);
    dq_kernel<D><<<static_cast<unsigned>(grid), 384, smem, s>>>(tq, tk, tv, tdo, p);
    timing_end(kKidDq, s);
    if (cudaGetLastError() != cudaSuccess) return LSX_ERR_LAUNCH;
  }
  return LSX_OK;
}

}  // namespace

int launch_bwd_tc(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                  const lsx_tensor& lse, const lsx_tensor& d_o, const float* delta,
                  int64_t q_off, int64_t kv_off, int causal, float scale,
                  const lsx_tensor& dq, const lsx_tensor& dk, const lsx_tensor& dv,
                  int accumulate, const DeviceCtx& ctx, cudaStream_t s) {
  if (q.D == 128)
    return launch_bwd_tc_d<128>(q, k, v, lse, d_o, delta, q_off, kv_off, causal, scale, dq, dk,
                                dv, accumulate, ctx, s);
  if (q.D == 64)
    return launch_bwd_tc_d<64>(q, k, v, lse, d_o, delta, q_off, kv_off, causal, scale, dq, dk,
                               dv, accumulate, ctx, s);
  return LSX_ERR_UNSUPPORTED;
}

}  // namespace lsx
