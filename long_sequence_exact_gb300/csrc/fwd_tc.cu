// fwd_tc.cu -- tcgen05 forward of exact attention over chunk pairs (bf16 in,
// fp32 accumulation in tensor memory).
//
// What it computes: for every query row i of a query chunk (absolute start
// q_off) against a key/value chunk (absolute start kv_off), the normalised
// output O_i = softmax(scale * q_i K^T) V over the visible keys and
// LSE_i = log sum_j exp(scale * <q_i, k_j>).  This is the "local attention
// computation" of BurstAttention (method section), evaluated with the online
// softmax whose associativity Lean Attention (abstract) relies on: a running
// row maximum m and sum l, with the output rescaled whenever m grows.
//
// Work decomposition (DistFlashAttn core concepts, load-balanced scheduling,
// with SMs as the workers): a persistent grid of one CTA per SM; a work item
// is two adjacent 128-row query tiles of one (batch, head); items are dealt
// longest-first in snake order.  Within an item the CTA walks every visible
// 128-key tile in order; crossing a key-chunk boundary simply continues the
// online softmax, which equals computing each chunk pair's partial and
// merging the partials in that order.
//
// CTA roles (384 threads):
//   warp 0        TMA producer: Q tiles once per item, K/V tiles through a
//                 ring of kStages stages (128-byte swizzle, zero fill past
//                 the end of a chunk).
//   warp 1        TMEM owner; lane 0 issues every tcgen05.mma:
//                 S_t = Q_t K^T   (SS, both K-major)            -> TMEM S_t
//                 O_t += P_t V    (TS, P_t from TMEM, V MN-major) -> TMEM O_t
//   warps 4..7    softmax of query tile 0 (thread = row = TMEM lane)
//   warps 8..11   softmax of query tile 1
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [384,384+D);
// P_t (bf16 pairs) overwrites the first 64 columns of S_t after the softmax
// has read S_t.  The MMA issue order per key tile j is
//   P_0 V_j, S_0(j+1), P_1 V_j, S_1(j+1)
// so each tile's softmax overlaps two MMAs of the other tile.  K and V slots
// are released separately (K after the S products, V after the P V ones).
// Softmax: all four TMEM loads in flight at once, 3-input max, packed fp32
// FMA/add (two elements per instruction) for the exp2 argument and row sum.
//
// Rescaling: the output is rescaled only when the row maximum grows by more
// than 8 (base 2); otherwise the stale maximum is kept, so exp2 arguments
// stay <= 8 (P <= 256), and the final O / l uses one consistent maximum, so
// the result is unchanged.
#include <cuda_bf16.h>
#include <math.h>

#include "fwd_split.h"
#include "internal.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace lsx {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile
  static constexpr int kSub = D / 64;             // 64-column (128 B) boxes
};

template <int D>
struct __align__(1024) FwdSmem {
  __nv_bfloat16 q[2][128 * D];
  __nv_bfloat16 k[FwdCfg<D>::kStages][128 * D];
  __nv_bfloat16 v[FwdCfg<D>::kStages][128 * D];
  uint64_t q_full, q_empty, final_bar;
  uint64_t k_full[FwdCfg<D>::kStages];
  uint64_t v_full[FwdCfg<D>::kStages];
  uint64_t k_empty[FwdCfg<D>::kStages];
  uint64_t v_empty[FwdCfg<D>::kStages];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint32_t tmem_base;
  int abort;
};

struct FwdParams {
  int64_t B, Hq, Hkv, Lq, Lk;
  int64_t q_off, kv_off;
  int causal, accumulate;
  float scale_log2;
  int64_t n_qpairs, n_items;
  void* o;
  int o_f32;
  int64_t o_sb, o_sh, o_sn;
  float* lse;
  int64_t l_sb, l_sh, l_sn;
  int* status;
  uint64_t wait_ns;
  // block-sparse lists (NULL: every key tile up to the causal limit)
  const int32_t* pair_count;
  const int32_t* pair_list;
  const uint8_t* bmask;  // [n_qtiles][n_kb]
  int64_t n_qtiles, n_kb;
  uint64_t* trace;  // per-CTA schedule record (NULL: not traced)
  // rows split into key pieces (piece_w 0: not split); n_items counts
  // kmax * n_qpairs * B * Hq items then, piece-major
  int64_t piece_w, kmax;
  float* part_o;    // [kmax][B][Hq][Lq][D] fp32
  float* part_lse;  // [kmax][B][Hq][Lq]
};

struct Item {
  int64_t b, h, hk, pair;
  int64_t nkv[2];  // key tiles this item visits for query tile 2 pair + t
};

// The piece of split rows an item is (kept apart from Item: its fields
// alone cost the unsplit kernel registers, even unused).
struct Piece {
  int64_t j0 = 0;     // position of its first key tile
  int64_t piece = 0;  // slot of its partials
  bool empty = false; // past the pair's last visible key tile: skipped
};

// (kSplit: rows split into key pieces; a template parameter, so that the
// unsplit kernel carries none of it)
template <bool kSplit>
__device__ __forceinline__ Item decode_item(const FwdParams& p, int64_t it, Piece* pc = nullptr) {
  Item x;
  if constexpr (kSplit) {
    // piece-major: every pair's first piece (pairs longest first), then
    // every pair's second, ...: full pieces come before a round's short and
    // empty ones, which the snake deal then spreads over the CTAs
    const int64_t per_piece = p.n_qpairs * p.B * p.Hq;
    pc->piece = it / per_piece;
    it -= pc->piece * per_piece;
  }
  int64_t rank, bh;
  banded_item(it, p.n_qpairs, p.B * p.Hq, &rank, &bh);
  x.pair = p.n_qpairs - 1 - rank;
  x.b = bh / p.Hq;
  x.h = bh % p.Hq;
  x.hk = x.h / (p.Hq / p.Hkv);
  for (int t = 0; t < 2; ++t)
    x.nkv[t] = p.pair_list == nullptr
                   ? fwd_kv_tiles(2 * x.pair + t, p.Lq, p.Lk, p.q_off, p.kv_off, p.causal)
                   : (2 * x.pair + t < p.n_qtiles ? p.pair_count[x.pair] : 0);
  if constexpr (kSplit) {
    pc->j0 = pc->piece * p.piece_w;
    pc->empty = pc->j0 >= (x.nkv[0] > x.nkv[1] ? x.nkv[0] : x.nkv[1]);
    for (int t = 0; t < 2; ++t) {
      const int64_t n = x.nkv[t] - pc->j0;
      x.nkv[t] = n < 0 ? 0 : (n > p.piece_w ? p.piece_w : n);
    }
  }
  return x;
}

// Key tile visited at position j of an item (the j-th listed tile when the
// attention is block-sparse).
__device__ __forceinline__ int64_t key_tile(const FwdParams& p, const Item& x, int64_t j,
                                            int64_t j0) {
  return p.pair_list == nullptr ? j0 + j : p.pair_list[x.pair * p.n_kb + j];
}

// Wait that ignores the abort flag but keeps the time bound (used at exit).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity,
                                           uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) break;
  }
}

template <int D, bool kVt, bool kSplit>
__global__ void __launch_bounds__(384, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const FwdParams p) {
  using Cfg = FwdCfg<D>;
  constexpr int kStages = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<D>& sm = *reinterpret_cast<FwdSmem<D>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitGuard guard{p.status, p.wait_ns, &sm.abort};

  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.final_bar, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm.s_full[t], 1);
      mbar_init(&sm.p_full[t], 128);
      mbar_init(&sm.o_full[t], 1);
    }
    fence_barrier_init();
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  if (p.trace != nullptr && threadIdx.x == 0)
    trace_begin(p.trace, kKidFwdTc, p.n_items, global_timer_ns());
  // 384 threads launched at <= 168 registers (64,512).  Producer/MMA
  // warpgroup keeps 104 (the issuing thread spills with less, and it is on
  // the critical path), the two softmax warpgroups take 200:
  // 128 * 104 + 256 * 200 = 64,512 <= 64,512.
  if (warp < 4) {
  regs_dec<104>();
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0, qe_phase = 0;
    int64_t r = 0;
    for (;; ++r) {
      const int64_t it = snake_item(c, r, G);
      if (it >= p.n_items) break;
      Piece pc;
      const Item x = decode_item<kSplit>(p, it, &pc);
      if (kSplit && pc.empty) continue;  // (every role skips the same items)
      const int64_t nkv = x.nkv[0] > x.nkv[1] ? x.nkv[0] : x.nkv[1];
      if (!mbar_wait(&sm.q_empty, qe_phase ^ 1, guard)) break;
      qe_phase ^= 1;
      mbar_arrive_expect_tx(&sm.q_full, 2 * Cfg::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int sub = 0; sub < Cfg::kSub; ++sub)
          tma_load_4d(&sm.q[t][sub * 128 * 64], &tm_q, &sm.q_full, sub * 64,
                      static_cast<int>((2 * x.pair + t) * 128),
                      static_cast<int>(x.h), static_cast<int>(x.b));
      bool ok = true;
      for (int64_t j = 0; j < nkv; ++j) {
        const int64_t kt = key_tile(p, x, j, kSplit ? pc.j0 : 0);
        if (!mbar_wait(&sm.k_empty[stage], phase ^ 1, guard)) { ok = false; break; }
        mbar_arrive_expect_tx(&sm.k_full[stage], Cfg::kTileBytes);
        for (int sub = 0; sub < Cfg::kSub; ++sub)
          tma_load_4d(&sm.k[stage][sub * 128 * 64], &tm_k, &sm.k_full[stage],
                      sub * 64, static_cast<int>(kt * 128),
                      static_cast<int>(x.hk), static_cast<int>(x.b));
        if (!mbar_wait(&sm.v_empty[stage], phase ^ 1, guard)) { ok = false; break; }
        mbar_arrive_expect_tx(&sm.v_full[stage], Cfg::kTileBytes);
        if constexpr (kVt) {
          // V^T tile: D rows (d) x 128 keys, as two 64-key boxes
          for (int sub = 0; sub < 2; ++sub)
            tma_load_4d(&sm.v[stage][sub * D * 64], &tm_v, &sm.v_full[stage],
                        static_cast<int>(kt * 128 + sub * 64), 0,
                        static_cast<int>(x.hk), static_cast<int>(x.b));
        } else {
          for (int sub = 0; sub < Cfg::kSub; ++sub)
            tma_load_4d(&sm.v[stage][sub * 128 * 64], &tm_v, &sm.v_full[stage],
                        sub * 64, static_cast<int>(kt * 128),
                        static_cast<int>(x.hk), static_cast<int>(x.b));
        }
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
    }
    if (p.trace != nullptr) trace_items(p.trace, r);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t kIdO = idesc_bf16_f32(128, D, 0, kVt ? 0 : 1);
    // Order per key tile j:  P_0 V_j, S_0 = Q_0 K_{j+1}^T, P_1 V_j, S_1 = ...
    // S_t(j+1) overwrites the TMEM columns that P_t(j) occupies; it is
    // issued right after P_t(j) V_j by this same thread, and one thread's
    // tcgen05.mma operations execute in issue order, so the P_t(j) reads of
    // the earlier MMA precede the S_t(j+1) writes of the later one.  This
    // gives each tile's softmax the time of two other MMAs (P_{1-t} V and
    // S_{1-t}) to finish before its P_t V is due.
    uint32_t kst = 0, kph = 0, vst = 0, vph = 0, q_phase = 0;
    uint32_t p_phase[2] = {0, 0};
    bool issued = false;
    const uint32_t q_addr[2] = {smem_addr(sm.q[0]), smem_addr(sm.q[1])};
    const uint64_t q_desc[2] = {sdesc_sw128(q_addr[0], 16, 1024),
                                sdesc_sw128(q_addr[1], 16, 1024)};
    auto issue_s = [&](int t, uint32_t k_addr) {
      const uint64_t k0 = sdesc_sw128(k_addr, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + t * 128, q_desc[t] + kmajor_step(kk, 128), k0 + kmajor_step(kk, 128),
               kIdS, kk > 0 ? 1u : 0u);
      mma_commit(&sm.s_full[t]);
    };
    for (int64_t r = 0;; ++r) {
      const int64_t it = snake_item(c, r, G);
      if (it >= p.n_items) break;
      Piece pc;
      const Item x = decode_item<kSplit>(p, it, &pc);
      if (kSplit && pc.empty) continue;
      const int64_t nkv = x.nkv[0] > x.nkv[1] ? x.nkv[0] : x.nkv[1];
      if (!mbar_wait(&sm.q_full, q_phase, guard)) break;
      q_phase ^= 1;
      tc_fence_after();
      bool ok = true;
      if (nkv > 0) {  // S_t(0)
        if (!mbar_wait(&sm.k_full[kst], kph, guard)) break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (x.nkv[t] > 0) issue_s(t, smem_addr(sm.k[kst]));
        issued = true;
        mma_commit(&sm.k_empty[kst]);
        if (++kst == kStages) { kst = 0; kph ^= 1; }
      }
      for (int64_t j = 0; j < nkv; ++j) {
        if (!mbar_wait(&sm.v_full[vst], vph, guard)) { ok = false; break; }
        tc_fence_after();
        const uint32_t v_addr = smem_addr(sm.v[vst]);
        const bool has_next = j + 1 < nkv;
        bool k_ready = false;
        for (int t = 0; t < 2; ++t) {
          if (j < x.nkv[t]) {
            if (!mbar_wait(&sm.p_full[t], p_phase[t], guard)) { ok = false; break; }
            p_phase[t] ^= 1;
            tc_fence_after();
            {
              // V^T: K-major (keys contiguous), 64-key boxes of D rows;
              // V: MN-major (d contiguous), 16 keys = 2048 bytes per step
              const uint64_t v0 = kVt ? sdesc_sw128(v_addr, 16, 1024)
                                      : sdesc_sw128(v_addr, 128 * 128, 1024);
              const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ts(tmem + 256 + t * 128, tmem + t * 128 + kk * 8,
                       v0 + (kVt ? kmajor_step(kk, D) : mnmajor_step(kk)), kIdO,
                       kk > 0 ? 1u : acc0);
            }
            mma_commit(&sm.o_full[t]);
          }
          if (has_next && j + 1 < x.nkv[t]) {
            if (!k_ready) {
              if (!mbar_wait(&sm.k_full[kst], kph, guard)) { ok = false; break; }
              tc_fence_after();
              k_ready = true;
            }
            issue_s(t, smem_addr(sm.k[kst]));
          }
        }
        if (!ok) break;
        if (has_next) {
          if (!k_ready) {  // K_{j+1} unused by both tiles: still consume its slot
            if (!mbar_wait(&sm.k_full[kst], kph, guard)) { ok = false; break; }
          }
          mma_commit(&sm.k_empty[kst]);
          if (++kst == kStages) { kst = 0; kph ^= 1; }
        }
        mma_commit(&sm.v_empty[vst]);
        if (++vst == kStages) { vst = 0; vph ^= 1; }
      }
      if (!ok) break;
      mma_commit(&sm.q_empty);
    }
    if (issued) {  // every issued MMA has completed before TMEM is released
      mma_commit(&sm.final_bar);
      drain_wait(&sm.final_bar, 0, p.wait_ns);
    }
  }
  } else {
    regs_inc<200>();
    // ------------------------------------------------------------- softmax
    const int t = (warp - 4) >> 2;
    const int row = threadIdx.x - 128 * (1 + t);  // 0..127 == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tO = tS + 256;
    uint32_t s_phase = 0;
    uint32_t pv_count = 0;
    const float sl2 = p.scale_log2;
    // The key-tile loop holds 128 scores in registers: keep little else live
    // across it (the item is decoded again for the epilogue, the wait guard
    // is rebuilt from the parameters at each wait, the grid position is
    // re-read), so that none of it spills.
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return mbar_wait(bar, parity, WaitGuard{p.status, p.wait_ns, &sm.abort});
    };
    for (int r = 0;; ++r) {
      const int64_t it = snake_item(blockIdx.x, r, gridDim.x);
      if (it >= p.n_items) break;
      int nkv;
      int64_t pair, j0 = 0;
      {
        Piece pc;
        const Item x = decode_item<kSplit>(p, it, &pc);
        if (kSplit && pc.empty) continue;
        nkv = static_cast<int>(x.nkv[t]);
        pair = x.pair;
        if constexpr (kSplit) j0 = pc.j0;
      }
      const int64_t qr0 = (2 * pair + t) * 128;
      float m = kNegInf, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        if (!wait(&sm.s_full[t], s_phase)) { ok = false; break; }
        s_phase ^= 1;
        tc_fence_after();
        float s[128];
        {
          // all four loads in flight before the single wait
          uint32_t u0[32], u1[32], u2[32], u3[32];
          tmem_ld32(tS, u0);
          tmem_ld32(tS + 32, u1);
          tmem_ld32(tS + 64, u2);
          tmem_ld32(tS + 96, u3);
          tmem_ld_wait32(u0);
          reg_fence32(u1);
          reg_fence32(u2);
          reg_fence32(u3);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(u0[i]);
            s[32 + i] = __uint_as_float(u1[i]);
            s[64 + i] = __uint_as_float(u2[i]);
            s[96 + i] = __uint_as_float(u3[i]);
          }
        }
        // (the key_tile position: j0 + j, or the j-th listed tile)
        const int64_t kb =
            (p.pair_list == nullptr ? (kSplit ? j0 + j : j) : p.pair_list[pair * p.n_kb + j]) *
            int64_t{128};
        // a listed tile whose block this query tile does not have: all masked
        const bool blk_off =
            p.bmask != nullptr && p.bmask[(2 * pair + t) * p.n_kb + kb / 128] == 0;
        const bool need_mask =
            blk_off || (kb + 128 > p.Lk) || (p.causal && p.kv_off + kb + 127 > p.q_off + qr0);
        if (need_mask) {
          int64_t lim = blk_off ? -1 : 127;
          if (kb + 128 > p.Lk && p.Lk - kb - 1 < lim) lim = p.Lk - kb - 1;
          if (p.causal) {
            const int64_t c2 = p.q_off + qr0 + row - p.kv_off - kb;
            if (c2 < lim) lim = c2;
          }
          const int climit = lim < -1 ? -1 : static_cast<int>(lim);
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i > climit) s[i] = kNegInf;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int i = 4; i < 128; i += 8) {
          mx0 = fmax3(mx0, s[i], s[i + 1]);
          mx1 = fmax3(mx1, s[i + 2], s[i + 3]);
          mx2 = fmax3(mx2, s[i + 4], s[i + 5]);
          mx3 = fmax3(mx3, s[i + 6], s[i + 7]);
        }
        const float mx = fmax3(fmaxf(mx0, mx1), mx2, mx3);
        const float m_new = fmaxf(m, mx * sl2);
        if (j == 0) {
          m = m_new;
        } else {
          const bool need = m_new > m + kRescaleThreshold;
          if (__any_sync(0xffffffffu, need)) {
            // O_t must hold the finished P_t V of the previous key tile
            if (!wait(&sm.o_full[t], (pv_count - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            const float alpha = (m == kNegInf) ? 0.f : ex2(m - m_new);
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t u[32];
              tmem_ld32(tO + cc * 32, u);
              tmem_ld_wait32(u);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
              tmem_st32(tO + cc * 32, u);
            }
            tmem_st_wait();
            l *= alpha;
            m = m_new;
          }
        }
        const float mu = (m == kNegInf) ? 0.f : m;
        // exp2(s * scale log2e - m) two at a time (packed fp32 FMA / add)
        const float2 sc2 = make_float2(sl2, sl2);
        const float2 nm2 = make_float2(-mu, -mu);
        float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 arg =
                __ffma2_rn(make_float2(s[cc * 32 + 2 * i], s[cc * 32 + 2 * i + 1]), sc2, nm2);
            const float2 e = make_float2(ex2(arg.x), ex2(arg.y));
            if (i & 1) lb = __fadd2_rn(lb, e); else la = __fadd2_rn(la, e);
            pk[i] = pack_bf16(e.x, e.y);
          }
          tmem_st16(tS + cc * 16, pk);
        }
        l += (la.x + la.y) + (lb.x + lb.y);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full[t]);
        ++pv_count;
      }
      if (!ok) break;
      // --------------------------------------------------------- epilogue
      Piece pc;
      const Item x = decode_item<kSplit>(p, it, &pc);
      const int64_t qrow = qr0 + row;
      const bool valid = qrow < p.Lq;
      // split rows: this piece's normalised partial goes to its fp32 slot
      int64_t prow = 0;
      if constexpr (kSplit) prow = ((pc.piece * p.B + x.b) * p.Hq + x.h) * p.Lq + qrow;
      if (nkv > 0) {
        if (!wait(&sm.o_full[t], (pv_count - 1) & 1)) break;
        tc_fence_after();
      }
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      float lse_new = (l > 0.f) ? (m + lg2(l)) * kLn2 : kNegInf;
      float w_old = 0.f, w_new = 1.f;
      if (p.accumulate && valid) {
        const float lse_old = p.lse[x.b * p.l_sb + x.h * p.l_sh + qrow * p.l_sn];
        const float mm = fmaxf(lse_old, lse_new);
        if (mm == kNegInf) {
          w_old = 0.f; w_new = 0.f;
        } else {
          const float wa = expf(lse_old - mm), wb = expf(lse_new - mm);
          const float tot = wa + wb;
          w_old = wa / tot; w_new = wb / tot;
          lse_new = mm + logf(tot);
        }
      }
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t u[32];
        if (nkv > 0) {
          tmem_ld32(tO + cc * 32, u);
          tmem_ld_wait32(u);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        if (!valid) continue;
        float ov[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) ov[i] = __uint_as_float(u[i]) * inv * w_new;
        int64_t base;
        if constexpr (kSplit)
          base = prow * D + cc * 32;
        else
          base = x.b * p.o_sb + x.h * p.o_sh + qrow * p.o_sn + cc * 32;
        if (kSplit || p.o_f32) {
          float* dst = (kSplit ? p.part_o : static_cast<float*>(p.o)) + base;
          if (p.accumulate) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 old = *reinterpret_cast<const float4*>(dst + i);
              ov[i] += w_old * old.x; ov[i + 1] += w_old * old.y;
              ov[i + 2] += w_old * old.z; ov[i + 3] += w_old * old.w;
            }
          }
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]);
        } else {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + base;
          if (p.accumulate) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              const uint4 old = *reinterpret_cast<const uint4*>(dst + i);
              const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&ow[e]);
                ov[i + 2 * e] += w_old * __low2float(pr);
                ov[i + 2 * e + 1] += w_old * __high2float(pr);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16(ov[i], ov[i + 1]);
            w.y = pack_bf16(ov[i + 2], ov[i + 3]);
            w.z = pack_bf16(ov[i + 4], ov[i + 5]);
            w.w = pack_bf16(ov[i + 6], ov[i + 7]);
            *reinterpret_cast<uint4*>(dst + i) = w;
          }
        }
      }
      if (valid) {
        if constexpr (kSplit)
          p.part_lse[prow] = lse_new;
        else
          p.lse[x.b * p.l_sb + x.h * p.l_sh + qrow * p.l_sn] = lse_new;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (p.trace != nullptr && threadIdx.x == 0) trace_end(p.trace, global_timer_ns());
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
int launch_fwd_tc_d(const lsx_tensor& q, const lsx_tensor& k,
                    const lsx_tensor& v, int64_t q_off, int64_t kv_off,
                    int causal, float scale, const lsx_tensor& o,
                    const lsx_tensor& lse, int accumulate, void* vt,
                    const DeviceCtx& ctx, cudaStream_t s, const BlockLists* bl,
                    const FwdSplit* split) {
  CUtensorMap tq, tk, tv;
  if (!make_map_bf16_4d(&tq, q.data, q.B, q.H, q.N, q.D, q.stride_b, q.stride_h,
                        q.stride_n, 128) ||
      !make_map_bf16_4d(&tk, k.data, k.B, k.H, k.N, k.D, k.stride_b, k.stride_h,
                        k.stride_n, 128))
    return LSX_ERR_LAUNCH;
  if (vt != nullptr) {
    // V^T [B, Hkv, D, Np]: rows are d, the inner (contiguous) axis is keys
    const int rc = launch_transpose(v, vt, s);
    if (rc != LSX_OK) return rc;
    const int64_t np = transposed_row_len(v.N);
    if (!make_map_bf16_4d(&tv, vt, v.B, v.H, v.D, v.N, v.H * v.D * np, v.D * np, np, D))
      return LSX_ERR_LAUNCH;
  } else if (!make_map_bf16_4d(&tv, v.data, v.B, v.H, v.N, v.D, v.stride_b, v.stride_h,
                               v.stride_n, 128)) {
    return LSX_ERR_LAUNCH;
  }
  FwdParams p;
  p.B = q.B; p.Hq = q.H; p.Hkv = k.H; p.Lq = q.N; p.Lk = k.N;
  p.q_off = q_off; p.kv_off = kv_off;
  p.causal = causal; p.accumulate = accumulate;
  p.scale_log2 = scale * kLog2e;
  p.n_qpairs = ceil_div(q.N, 256);
  p.n_items = p.n_qpairs * q.B * q.H;
  p.o = o.data; p.o_f32 = (o.dtype == LSX_F32);
  p.o_sb = o.stride_b; p.o_sh = o.stride_h; p.o_sn = o.stride_n;
  p.lse = static_cast<float*>(lse.data);
  p.l_sb = lse.stride_b; p.l_sh = lse.stride_h; p.l_sn = lse.stride_n;
  p.status = ctx.status; p.wait_ns = ctx.wait_ns;
  p.n_qtiles = ceil_div(q.N, 128);
  p.pair_count = bl ? bl->pair_count : nullptr;
  p.pair_list = bl ? bl->pair_list : nullptr;
  p.bmask = bl ? bl->mask : nullptr;
  p.n_kb = bl ? bl->n_kb : 0;
  p.piece_w = 0;
  p.kmax = 1;
  p.part_o = nullptr;
  p.part_lse = nullptr;
  if (split != nullptr && split->piece_w > 0) {
    // (never with block lists or accumulation: the chunked call alone splits)
    if (bl != nullptr || accumulate || split->kmax < 1) return LSX_ERR_UNSUPPORTED;
    p.piece_w = split->piece_w;
    p.kmax = split->kmax;
    p.part_o = split->part_o;
    p.part_lse = split->part_lse;
    p.n_items *= p.kmax;
  }
  const size_t smem = sizeof(FwdSmem<D>) + 1024;
  auto kern = p.piece_w > 0 ? (vt != nullptr ? fwd_tc_kernel<D, true, true>
                                             : fwd_tc_kernel<D, false, true>)
                           : (vt != nullptr ? fwd_tc_kernel<D, true, false>
                                            : fwd_tc_kernel<D, false, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return LSX_ERR_LAUNCH;
  const int64_t grid = p.n_items < ctx.sm_count ? p.n_items : ctx.sm_count;
  p.trace = trace_record(kKidFwdTc, grid);
  timing_begin(kKidFwdTc, s);
  kern<<<static_cast<unsigned>(grid), 384, smem, s>>>(tq, tk, tv, p);
  timing_end(kKidFwdTc, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

}  // namespace

size_t fwd_tc_workspace_bytes(const lsx_tensor& v) { return transposed_bytes(v); }

int launch_fwd_tc(const lsx_tensor& q, const lsx_tensor& k,
                  const lsx_tensor& v, int64_t q_off, int64_t kv_off,
                  int causal, float scale, const lsx_tensor& o,
                  const lsx_tensor& lse, int accumulate, void* vt,
                  const DeviceCtx& ctx, cudaStream_t s, const BlockLists* bl) {
  if (q.D == 128)
    return launch_fwd_tc_d<128>(q, k, v, q_off, kv_off, causal, scale, o, lse,
                                accumulate, vt, ctx, s, bl, nullptr);
  if (q.D == 64)
    return launch_fwd_tc_d<64>(q, k, v, q_off, kv_off, causal, scale, o, lse,
                               accumulate, vt, ctx, s, bl, nullptr);
  return LSX_ERR_UNSUPPORTED;
}

int launch_fwd_tc_split(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                        int64_t q_off, int64_t kv_off, int causal, float scale,
                        const lsx_tensor& o, const lsx_tensor& lse, void* vt,
                        const FwdSplit& split, const DeviceCtx& ctx, cudaStream_t s) {
  if (split.piece_w <= 0) return LSX_ERR_UNSUPPORTED;
  if (q.D == 128)
    return launch_fwd_tc_d<128>(q, k, v, q_off, kv_off, causal, scale, o, lse, 0, vt, ctx, s,
                                nullptr, &split);
  if (q.D == 64)
    return launch_fwd_tc_d<64>(q, k, v, q_off, kv_off, causal, scale, o, lse, 0, vt, ctx, s,
                               nullptr, &split);
  return LSX_ERR_UNSUPPORTED;
}

}  // namespace lsx
