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
// Persistent kernels:
//  * dkdv_kernel, key-tile-major: a work item is one 128-row key/value tile
//    of one (batch, kv head); it walks every query tile (of every query head
//    of the group) that sees it:
//      S^T  = K Q_i^T     (SS, K-major x K-major)      TMEM [0,128)
//      dP^T = V dO_i^T    (SS)                         TMEM [128,256)
//      grad warps: P^T once S^T is in, dS^T once dP^T is in, each as bf16
//      back into the first 16 columns of the warp's quarter of its tile
//      dV  += P^T dO_i    (TS, dO_i MN-major)          TMEM [256,256+D)
//      dK  += dS^T Q_i    (TS, Q_i MN-major)           TMEM [384,384+D)
//    dV is issued as soon as P^T is stored, so it runs while dS^T is
//    formed; dK once dS^T is.
//    With kDq and D = 128 it also forms dQ: once dV has read dO_i for the
//    last time, the grad warps write dS^T into dO_i's shared-memory slot and
//      dQ_i^T = K^T dS^T  (SS, both MN-major)          TMEM [128,256)
//    which they read back (the next dP^T waits only for that), scale and
//    stage in the now dead Q_i / dO_i slots; one thread of warp 2 adds the
//    staged tile into the fp32 dQ accumulator with TMA reduce-adds and frees
//    the slots for the next loads once the TMA unit has read them.  dK and
//    dV stay owned by one CTA each; dQ's summation order varies between
//    runs.
//    With kDq and D = 64, TMEM has room to spare and shared memory too:
//      dQ_i = dS K        (SS, both MN-major)     TMEM [320,384) / [448,512)
//    alternating between the two free 64-column regions, issued by a second
//    MMA thread (warp 3) from dS^T's own double-buffered shared tile, which
//    the grad warps write after publishing P^T and dS^T.  That thread also
//    issues dK_i, in parallel with the first thread's dV_i; the first thread
//    issues step i+1's S^T right after dV_i (the last reader of its
//    columns) and its dP^T once dK_i has completed (dk_done), so dQ_i runs
//    under the grad warps' next step.  During step i+1 the grad warps read dQ_i back and stage it,
//    scaled, in dS_i^T's spent tile as two swizzled [128 queries][32 d]
//    fp32 boxes; one thread of warp 2 adds them into the target with
//    tensor-map reduce-adds and releases the tile for the dS^T of step i+2.
//    (Where the target takes no tensor map the grad warps add with 16-byte
//    vector atomics instead.)
//  * dq_kernel (the deterministic form of dQ), query-tile-major: a work item
//    is one 128-row query tile; it walks every visible key tile:
//      S  = Q K_j^T, dP = dO V_j^T (SS)                TMEM [0,128), [128,256)
//      grad warps: dS -> bf16 into TMEM (inside [128,256))
//      dQ += dS K_j       (TS, K_j MN-major)           TMEM [256,256+D)
// Roles per CTA (640 threads): warp 0 loads (TMA), warp 1 owns TMEM and
// issues the MMAs (lane 0; with fused dQ at D = 64, warp 3 issues the dK
// and dQ products), warp 2 (lane 0) adds the staged dQ into its target, and the 16
// grad warps 4..19 compute P and dS and write the outputs.  Grad warp g
// covers TMEM lanes 32 (g % 4) .. +31 and the quarter g / 4 of the 128
// columns; each quarter packs its bf16 result into its own first 16
// columns, so warps sharing a lane range never touch each other's columns,
// and the TS MMAs address each 16-wide K step of the bf16 operand at
// packed_col(kk).
// MMA issue order: products of one thread execute in issue order, so a
// product that overwrites TMEM columns is issued after the products that
// read them (e.g. the next S^T after the dV that reads P^T); products of
// the two issuing threads touch disjoint columns and are ordered by
// barriers.  Work items are dealt longest-first in snake order.
#include <cuda_bf16.h>
#include <math.h>

#include "bwd_split.h"
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
  // block-sparse lists (NULL: dense tile ranges up to the causal limit)
  const int32_t* row_count;
  const int32_t* row_list;  // stride n_ktiles
  const int32_t* col_count;
  const int32_t* col_list;  // stride n_qtiles
  // fused dQ: fp32 accumulator and its strides (elements); with acc_tma it
  // is added into through the tensor map tm_acc: at D = 128 the accumulator
  // is transposed, [B][Hq][128][Np]; at D = 64 it is [B][Hq][N][64] with the
  // strides above (boxes of [128 queries][32 d])
  float* dq_acc;
  int64_t acc_sb, acc_sh, acc_sn;
  int acc_tma;
  uint64_t* trace;  // per-CTA schedule record (NULL: not traced)
  int trace_kid;
  // fused dK/dV with key columns split into pieces of piece_w steps (the
  // dkdv kernel's kSplit form): piece i of every item writes its partial
  // dK, dV (fp32) to slot i of part_dk / part_dv [kmax][B][Hkv][Lk][D]
  int64_t piece_w, kmax;
  float* part_dk;
  float* part_dv;
};

// Row pitch (elements) of the transposed fp32 dQ accumulator [.][128][Np]:
// N rounded up to 16-byte rows, as tensor maps require.
__host__ __device__ inline int64_t dq_acc_pitch(int64_t n) { return (n + 3) / 4 * 4; }

// TMEM column (relative to the 128-column fp32 tile) of the packed bf16
// operand for K step kk (16 elements = 8 packed columns).
__device__ __forceinline__ uint32_t packed_col(int kk) {
  return static_cast<uint32_t>(32 * (kk >> 1) + 8 * (kk & 1));
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

// Loads 32 fp32 columns of two TMEM tiles with one wait.
__device__ __forceinline__ void ld_two(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                       uint32_t (&b)[32]) {
  tmem_ld32(ta, a);
  tmem_ld32(tb, b);
  tmem_ld_wait32(a);
  reg_fence32(b);
}

// P^T and dS^T of one grad thread's 32 scores when the score products
// already hold S - LSE/scale and dP - delta; with kMask, the query columns
// c < cmin (not yet visible to this key) get P = 0.  Formed in two halves,
// so that P^T can be computed as soon as S^T is in, while dP^T is still
// being computed: P of the 32 scores (kept in fp32 for dS, and packed to
// bf16 for the dV product) ...
template <bool kMask>
__device__ __forceinline__ void p_rows_rs(const uint32_t (&us)[32], float2 sc2, int cmin,
                                          float (&pr)[32], uint32_t (&pk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int c0 = 2 * e;
    const float2 arg = __fmul2_rn(
        make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sc2);
    float2 v = make_float2(ex2(arg.x), ex2(arg.y));
    if (kMask) {
      if (c0 < cmin) v.x = 0.f;
      if (c0 + 1 < cmin) v.y = 0.f;
    }
    pr[c0] = v.x;
    pr[c0 + 1] = v.y;
    pk[e] = pack_bf16(v.x, v.y);
  }
}
// ... and dS^T = P^T o (dP^T - delta) once dP^T is in.
__device__ __forceinline__ void ds_rows_rs(const float (&pr)[32], const uint32_t (&ud)[32],
                                           uint32_t (&dk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float2 ds = __fmul2_rn(make_float2(pr[2 * e], pr[2 * e + 1]),
                                 make_float2(__uint_as_float(ud[2 * e]),
                                             __uint_as_float(ud[2 * e + 1])));
    dk[e] = pack_bf16(ds.x, ds.y);
  }
}
// Without the statistics on the tensor cores: LSE (log2 units) and delta of
// the 32 query columns come from shared memory.
__device__ __forceinline__ void p_rows_st(const uint32_t (&us)[32], float2 sc2,
                                          const float4* l2v, int cmin, float (&pr)[32],
                                          uint32_t (&pk)[16]) {
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 l4 = l2v[e4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int e = e4 * 2 + hh;
      const int c0 = 2 * e;
      const float2 nl = hh ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
      const float2 arg = __ffma2_rn(
          make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sc2, nl);
      float2 v = make_float2(ex2(arg.x), ex2(arg.y));
      if (c0 < cmin) v.x = 0.f;
      if (c0 + 1 < cmin) v.y = 0.f;
      pr[c0] = v.x;
      pr[c0 + 1] = v.y;
      pk[e] = pack_bf16(v.x, v.y);
    }
  }
}
__device__ __forceinline__ void ds_rows_st(const float (&pr)[32], const uint32_t (&ud)[32],
                                           const float4* dlv, uint32_t (&dk)[16]) {
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const float4 d4 = dlv[e4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int e = e4 * 2 + hh;
      const float2 nd = hh ? make_float2(-d4.z, -d4.w) : make_float2(-d4.x, -d4.y);
      const float2 dpm = __fadd2_rn(
          make_float2(__uint_as_float(ud[2 * e]), __uint_as_float(ud[2 * e + 1])), nd);
      const float2 ds = __fmul2_rn(make_float2(pr[2 * e], pr[2 * e + 1]), dpm);
      dk[e] = pack_bf16(ds.x, ds.y);
    }
  }
}

// dS of one dQ grad thread's 32 scores; with kMask, key columns c > climit
// (not visible to this query, or past the keys) get P = 0.
template <bool kMask>
__device__ __forceinline__ void grad_cols_dq(const uint32_t (&us)[32], const uint32_t (&ud)[32],
                                             float2 sc2, float2 nl, float2 nd, int climit,
                                             uint32_t (&dk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const int c0 = 2 * e;
    const float2 arg = __ffma2_rn(
        make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])), sc2, nl);
    float2 pr = make_float2(ex2(arg.x), ex2(arg.y));
    if (kMask) {
      if (c0 > climit) pr.x = 0.f;
      if (c0 + 1 > climit) pr.y = 0.f;
    }
    const float2 dpm = __fadd2_rn(
        make_float2(__uint_as_float(ud[2 * e]), __uint_as_float(ud[2 * e + 1])), nd);
    const float2 ds = __fmul2_rn(pr, dpm);
    dk[e] = pack_bf16(ds.x, ds.y);
  }
}

// ===================================================================== dK dV
// The dV / dK products read dO and Q as stored (MN-major B operands, the
// same tiles the S^T / dP^T products use): measured faster here than
// loading sequence-contiguous copies, whose extra shared-memory traffic
// slows the SS products more than the K-major reads gain.
template <int D>
struct DkdvSmem {
  __nv_bfloat16 k[128 * D];
  __nv_bfloat16 v[128 * D];
  __nv_bfloat16 q[2][128 * D];
  __nv_bfloat16 d_o[2][128 * D];
  __nv_bfloat16 rs[2][128 * 8];   // row statistics of Q_i (core-matrix order)
  __nv_bfloat16 ones[2][128 * 8]; // selector tiles for -LSE/scale and -delta
  float lse2[2][128];             // LSE * log2(e); +inf for rows without keys
  float delta[2][128];
  uint64_t kv_full, kv_empty, final_bar, ones_full;
  uint64_t final_dq;  // D = 64 fused: the dQ issuer's last products are complete
  uint64_t q_full[2], q_empty[2], o_full[2], o_empty[2];  // Q_i (+ statistics), dO_i slots
  uint64_t lse_full[2], lse_empty[2];
  uint64_t s_ready, s_full, p_full, dkv_done;  // S^T in; S^T and dP^T in; P^T, dS^T out
  uint64_t pt_full;  // P^T out (dV may start while dS^T is being formed)
  uint64_t dv_done, ds_full, dq_full, dq_drained, stage_full;  // fused dQ, D = 128
  uint64_t dq_done[2], dq_free[2];                             // fused dQ, D = 64
  uint64_t ds_ready[2];  // D = 64: the dS^T tile of that parity has been written
  uint64_t dk_done;      // D = 64 fused: this step's dK (second issuer) has completed
  uint64_t stage_free[2];  // D = 64 with acc_tma: the dS^T tile's staged dQ has been read
  uint32_t tmem_base;
  int abort;
  // dS^T tiles of the D = 64 fused form (128-byte swizzle: 1024-aligned)
  alignas(1024) __nv_bfloat16 ds[D == 64 ? 2 : 1][D == 64 ? 128 * 128 : 8];
};

struct DkdvItem {
  int64_t b, hk, j, i0, n_i, group;
  int64_t len;  // query tiles per head of the group
};

// The piece of a split item (kept apart from DkdvItem, which the unsplit
// kernel keeps in registers).
struct DkdvPiece {
  int64_t s0 = 0;     // first step of the piece
  int64_t piece = 0;  // slot of its partials
  bool empty = false; // past the item's last step: skipped by every role
};

template <bool kSplit>
__device__ __forceinline__ DkdvItem dkdv_item(const BwdParams& p, int64_t it,
                                              DkdvPiece* pc = nullptr) {
  DkdvItem x;
  if constexpr (kSplit) {
    // piece-major: every item's first piece (longest first), then every
    // item's second, ...
    const int64_t per_piece = p.n_ktiles * p.B * p.Hkv;
    pc->piece = it / per_piece;
    it -= pc->piece * per_piece;
  }
  int64_t rank, bh;
  banded_item(it, p.n_ktiles, p.B * p.Hkv, &rank, &bh);
  x.j = rank;  // key tile 0 (the most query tiles) first
  x.b = bh / p.Hkv;
  x.hk = bh % p.Hkv;
  x.group = p.Hq / p.Hkv;
  x.i0 = q_tile_begin(p, x.j);
  x.len = p.col_list == nullptr ? p.n_qtiles - x.i0 : p.col_count[x.j];
  x.n_i = x.len * x.group;  // (head, query tile) steps
  if constexpr (kSplit) {
    pc->s0 = pc->piece * p.piece_w;
    pc->empty = pc->s0 >= x.n_i;
    const int64_t n = x.n_i - pc->s0;
    x.n_i = n < 0 ? 0 : (n > p.piece_w ? p.piece_w : n);
  }
  return x;
}

// The steps of a dK/dV item in order: every query tile of the group's
// first head, then of the next head.  A cursor advanced once per step (a
// 64-bit division per step would cost each thread that walks the item a
// few hundred cycles).
struct DkdvCursor {
  int64_t h, r;  // query head; position among the item's query tiles of a head
};
__device__ __forceinline__ DkdvCursor dkdv_first(const DkdvItem& x) {
  return DkdvCursor{x.hk * x.group, 0};
}
// ... and at step s0 (the first step of a piece: one division per item)
__device__ __forceinline__ DkdvCursor dkdv_at(const DkdvItem& x, int64_t s0) {
  return DkdvCursor{x.hk * x.group + s0 / x.len, s0 % x.len};
}
// Query head and query tile of the cursor's step, then on to the next step.
__device__ __forceinline__ void dkdv_take(const BwdParams& p, const DkdvItem& x, DkdvCursor& cur,
                                          int64_t& h, int64_t& i) {
  h = cur.h;
  i = p.col_list == nullptr ? x.i0 + cur.r : p.col_list[x.j * p.n_qtiles + cur.r];
  if (++cur.r == x.len) {
    cur.r = 0;
    ++cur.h;
  }
}

// Loads one 128-row tile as D/64 boxes of [128 rows][64 cols] (row-major
// view, d contiguous) or, from a transposed copy, two boxes of
// [D rows][64 sequence positions] (sequence contiguous).
template <int D, bool kTransposed>
__device__ __forceinline__ void load_tile(__nv_bfloat16* dst, const CUtensorMap* map,
                                          uint64_t* bar, int64_t row0, int64_t h, int64_t b) {
  if constexpr (kTransposed) {
    for (int sub = 0; sub < 2; ++sub)
      tma_load_4d(dst + sub * D * 64, map, bar, static_cast<int>(row0 + sub * 64), 0,
                  static_cast<int>(h), static_cast<int>(b));
  } else {
    for (int sub = 0; sub < D / 64; ++sub)
      tma_load_4d(dst + sub * 128 * 64, map, bar, sub * 64, static_cast<int>(row0),
                  static_cast<int>(h), static_cast<int>(b));
  }
}

// S-type product D (+)= A B^T over K = D, both operands K-major 128-row
// tiles; base descriptors are built once and stepped by constants so that
// the single issuing thread keeps ahead of the tensor pipe.
template <int D>
__device__ __forceinline__ void mma_rows_by_rows(uint32_t d_tmem, uint32_t a_addr,
                                                 uint32_t b_addr, uint32_t idesc) {
  const uint64_t a0 = sdesc_sw128(a_addr, 16, 1024);
  const uint64_t b0 = sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    mma_ss(d_tmem, a0 + kmajor_step(kk, 128), b0 + kmajor_step(kk, 128), idesc,
           kk > 0 ? 1u : 0u);
}

// Base descriptor and per-step offset of a B operand spanning a 128-row
// tile of the sequence: K-major from a transposed tile (D rows of 128
// positions), MN-major from the row-major tile.
template <int D, bool kTransposed>
__device__ __forceinline__ uint64_t seq_b_base(uint32_t base) {
  return kTransposed ? sdesc_sw128(base, 16, 1024) : sdesc_sw128(base, 128 * 128, 1024);
}
template <int D, bool kTransposed>
__host__ __device__ constexpr uint64_t seq_b_step(int kk) {
  return kTransposed ? kmajor_step(kk, D) : mnmajor_step(kk);
}

// With kRS the score products carry the row statistics themselves: after
// the D/16 K steps of K Q_i^T (or V dO_i^T) one more K step multiplies a
// selector tile by the statistics tile of Q_i, which adds -LSE/scale (or
// -delta) to every score of each query column; the grad warps then need
// neither the LSE nor delta.  Without kRS warp 0 gathers both into shared
// memory and the grad warps apply them per element.
template <int D, bool kRS, bool kDq, bool kSplit = false>
__global__ void __launch_bounds__(640, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_rs,
                const __grid_constant__ CUtensorMap tm_ones,
                const __grid_constant__ CUtensorMap tm_acc, const BwdParams p) {
  using Sm = DkdvSmem<D>;
  static_assert(!kDq || D == 128 || D == 64, "fused dQ: d = 128 or 64");
  constexpr bool kQ128 = kDq && D == 128;  // dQ^T in the dP^T columns, staged, bulk-reduced
  constexpr bool kQ64 = kDq && D == 64;    // dQ in free columns, staged in the spent dS^T tile
  constexpr int kTile = 128 * D * 2;
  constexpr int kQoStages = 2;
  extern __shared__ uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                  ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitGuard guard{p.status, p.wait_ns, &sm.abort};
  if (threadIdx.x == 0) {
    sm.abort = 0;
    mbar_init(&sm.kv_full, 1);
    // (D = 64 fused: K_j is also read by the dQ products of the second
    // issuing thread, which releases the slot too)
    mbar_init(&sm.kv_empty, kQ64 ? 2 : 1);
    mbar_init(&sm.final_bar, 1);
    mbar_init(&sm.final_dq, 1);
    mbar_init(&sm.ones_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.q_full[s], 1);
      mbar_init(&sm.q_empty[s], 1);
      mbar_init(&sm.o_full[s], 1);
      mbar_init(&sm.o_empty[s], 1);
      mbar_init(&sm.lse_full[s], 32);
      mbar_init(&sm.lse_empty[s], 512);
    }
    mbar_init(&sm.s_ready, 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, 512);
    mbar_init(&sm.pt_full, 512);
    mbar_init(&sm.dk_done, 1);
    mbar_init(&sm.dkv_done, 1);
    mbar_init(&sm.dv_done, 1);
    mbar_init(&sm.ds_full, 512);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_drained, 512);
    mbar_init(&sm.stage_full, 512);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.ds_ready[b], 512);
      mbar_init(&sm.dq_done[b], 1);
      mbar_init(&sm.dq_free[b], 512);
      mbar_init(&sm.stage_free[b], 1);
    }
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
  if (p.trace != nullptr && threadIdx.x == 0)
    trace_begin(p.trace, p.trace_kid, p.n_items, global_timer_ns());

  // 640 threads launched at <= 96 registers (61,440): the load/MMA
  // warpgroup keeps 64, the four grad warpgroups take 104:
  // 128 * 64 + 512 * 104 = 61,440 <= 61,440.
  if (warp < 4) {
    regs_dec<64>();
    if (warp == 0) {
      // -------------------------------------------------- loads (warp 0)
      uint32_t qs = 0, qph = 0, ls = 0, lph = 0, kv_phase = 0;
      if (kRS && lane == 0) {
        mbar_arrive_expect_tx(&sm.ones_full, 2 * 128 * 16);
        tma_load_4d(sm.ones[0], &tm_ones, &sm.ones_full, 0, 0, 0, 0);
        tma_load_4d(sm.ones[1], &tm_ones, &sm.ones_full, 0, 128, 0, 0);
      }
      int64_t r = 0;
      for (;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        DkdvPiece pc;
        const DkdvItem x = dkdv_item<kSplit>(p, it, &pc);
        if (kSplit && pc.empty) continue;  // (every role skips the same items)
        if (!mbar_wait(&sm.kv_empty, kv_phase ^ 1, guard)) break;
        kv_phase ^= 1;
        if (lane == 0) {
          mbar_arrive_expect_tx(&sm.kv_full, 2 * kTile);
          load_tile<D, false>(sm.k, &tm_k, &sm.kv_full, x.j * 128, x.hk, x.b);
          load_tile<D, false>(sm.v, &tm_v, &sm.kv_full, x.j * 128, x.hk, x.b);
        }
        bool ok = true;
        DkdvCursor cur = kSplit ? dkdv_at(x, pc.s0) : dkdv_first(x);
        for (int64_t s = 0; s < x.n_i; ++s) {
          int64_t h, i;
          dkdv_take(p, x, cur, h, i);
          // Q_i, dO_i (B operands of S^T, dP^T and, read MN-major, of dK, dV);
          // the two slots are freed separately (the fused form frees Q_i's
          // first) and S^T waits only for Q_i
          if (!mbar_wait(&sm.q_empty[qs], qph ^ 1, guard)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(&sm.q_full[qs], kTile + (kRS ? 128 * 16 : 0));
            load_tile<D, false>(sm.q[qs], &tm_q, &sm.q_full[qs], i * 128, h, x.b);
            if constexpr (kRS)
              tma_load_4d(sm.rs[qs], &tm_rs, &sm.q_full[qs], 0, static_cast<int>(i * 128),
                          static_cast<int>(h), static_cast<int>(x.b));
          }
          if (!mbar_wait(&sm.o_empty[qs], qph ^ 1, guard)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(&sm.o_full[qs], kTile);
            load_tile<D, false>(sm.d_o[qs], &tm_do, &sm.o_full[qs], i * 128, h, x.b);
          }
          if (++qs == kQoStages) { qs = 0; qph ^= 1; }
          if constexpr (kRS) continue;
          // LSE (log2 units) and delta of the 128 query rows of tile i
          if (!mbar_wait(&sm.lse_empty[ls], lph ^ 1, guard)) { ok = false; break; }
          for (int t = lane; t < 128; t += 32) {
            const int64_t row = i * 128 + t;
            float l2 = kPosInf, dl = 0.f;
            if (row < p.Lq) {
              const float lse = p.lse[x.b * p.l_sb + h * p.l_sh + row * p.l_sn];
              l2 = (lse == kNegInf) ? kPosInf : lse * kLog2e;
              dl = p.delta[(x.b * p.Hq + h) * p.Lq + row];
            }
            sm.lse2[ls][t] = l2;
            sm.delta[ls][t] = dl;
          }
          mbar_arrive(&sm.lse_full[ls]);
          if (++ls == 2) { ls = 0; lph ^= 1; }
        }
        if (!ok) break;
      }
      if (p.trace != nullptr && lane == 0) trace_items(p.trace, r);
    } else if (warp == 1 && lane == 0) {
      // ----------------------------------------------------------- MMA issue
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, 1);
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, 128, 1, 1);  // dQ^T = K^T dS^T
      uint32_t qs = 0, qph = 0, kv_phase = 0, p_phase = 0, ds_phase = 0, dr_phase = 0;
      uint32_t dk_phase = 0;
      bool issued = false, dq_pending = false;
      const uint32_t k_addr = smem_addr(sm.k), v_addr = smem_addr(sm.v);
      // selector and statistics tiles: 16 core matrices of 8 rows x 16 bytes
      // along M/N (128 bytes apart); the K step's second core matrix re-reads
      // the first (distance 0 along K), which the halved statistics undo.
      const uint64_t sel_c = sdesc_interleave(smem_addr(sm.ones[0]), 0, 128);
      const uint64_t sel_d = sdesc_interleave(smem_addr(sm.ones[1]), 0, 128);
      bool ones_ok = true;
      if constexpr (kRS) ones_ok = mbar_wait(&sm.ones_full, 0, guard);
      for (int64_t r = 0; ones_ok; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        DkdvPiece pc;
        const DkdvItem x = dkdv_item<kSplit>(p, it, &pc);
        if (kSplit && pc.empty) continue;  // (every role skips the same items)
        if (!mbar_wait(&sm.kv_full, kv_phase, guard)) break;
        kv_phase ^= 1;
        tc_fence_after();
        bool ok = true;
        for (int64_t s = 0; s < x.n_i; ++s) {
          const uint32_t q_addr = smem_addr(sm.q[qs]);
          const uint32_t o_addr = smem_addr(sm.d_o[qs]);
          // (kQ64: the S^T / dP^T of steps after an item's first were issued
          // by the step before, ahead of its dQ)
          if (!(kQ64 && s > 0)) {
            if (!mbar_wait(&sm.q_full[qs], qph, guard)) { ok = false; break; }
            tc_fence_after();
            const uint64_t st = sdesc_interleave(smem_addr(sm.rs[qs]), 0, 128);
            mma_rows_by_rows<D>(tmem + 0, k_addr, q_addr, kIdS);
            if constexpr (kRS) mma_ss(tmem + 0, sel_c, st, kIdS, 1u);
            mma_commit(&sm.s_ready);
            if (kQ128 && dq_pending) {  // dP^T reuses the columns of the last dQ^T
              if (!mbar_wait(&sm.dq_drained, dr_phase, guard)) { ok = false; break; }
              dr_phase ^= 1;
            }
            if (!mbar_wait(&sm.o_full[qs], qph, guard)) { ok = false; break; }
            tc_fence_after();
            mma_rows_by_rows<D>(tmem + 128, v_addr, o_addr, kIdS);
            if constexpr (kRS) mma_ss(tmem + 128, sel_d, st, kIdS, 1u);
            mma_commit(&sm.s_full);
            issued = true;
          }
          // dV += P^T dO_i as soon as P^T is in TMEM (pt_full): it runs while
          // the grad warps form dS^T; dK waits for that (p_full)
          if (!mbar_wait(&sm.pt_full, p_phase, guard)) { ok = false; break; }
          const uint32_t bq = q_addr, bo = o_addr;
          tc_fence_after();
          const uint64_t bo0 = seq_b_base<D, false>(bo), bq0 = seq_b_base<D, false>(bq);
          const uint32_t acc0 = s > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + 256, tmem + packed_col(kk), bo0 + seq_b_step<D, false>(kk), kIdG,
                   kk > 0 ? 1u : acc0);
          if constexpr (kQ128) mma_commit(&sm.dv_done);  // dO_i has been read for the last time
          if constexpr (kQ64) {
            // dK_i is issued by the second MMA thread (warp 3), in parallel
            // with dV_i here.  dO_i has been read for the last time (dP^T,
            // dV); Q_i's slot is released by that thread after dK_i.
            p_phase ^= 1;
            mma_commit(&sm.o_empty[qs]);
            // The next S^T right away: dV_i, the last reader of its columns
            // (P^T), precedes it in this thread's issue order.  The next dP^T
            // overwrites dS^T_i, which dK_i reads: it waits for dK_i.
            const bool next = s + 1 < x.n_i;
            const uint32_t ns = qs + 1 == kQoStages ? 0u : qs + 1;
            const uint32_t nph = qs + 1 == kQoStages ? qph ^ 1u : qph;
            if (next) {
              if (!mbar_wait(&sm.q_full[ns], nph, guard)) { ok = false; break; }
              tc_fence_after();
              const uint64_t nst = sdesc_interleave(smem_addr(sm.rs[ns]), 0, 128);
              mma_rows_by_rows<D>(tmem + 0, k_addr, smem_addr(sm.q[ns]), kIdS);
              if constexpr (kRS) mma_ss(tmem + 0, sel_c, nst, kIdS, 1u);
              mma_commit(&sm.s_ready);
            }
            if (!mbar_wait(&sm.dk_done, dk_phase, guard)) { ok = false; break; }
            dk_phase ^= 1;
            tc_fence_after();
            if (next) {
              if (!mbar_wait(&sm.o_full[ns], nph, guard)) { ok = false; break; }
              tc_fence_after();
              const uint64_t nst = sdesc_interleave(smem_addr(sm.rs[ns]), 0, 128);
              mma_rows_by_rows<D>(tmem + 128, v_addr, smem_addr(sm.d_o[ns]), kIdS);
              if constexpr (kRS) mma_ss(tmem + 128, sel_d, nst, kIdS, 1u);
              mma_commit(&sm.s_full);
            }
            if (++qs == kQoStages) { qs = 0; qph ^= 1; }
            continue;
          }
          if (!mbar_wait(&sm.p_full, p_phase, guard)) { ok = false; break; }
          p_phase ^= 1;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + 384, tmem + 128 + packed_col(kk), bq0 + seq_b_step<D, false>(kk), kIdG,
                   kk > 0 ? 1u : acc0);
          if constexpr (kQ128) {
            if (!mbar_wait(&sm.ds_full, ds_phase, guard)) { ok = false; break; }
            ds_phase ^= 1;
            tc_fence_after();
            // A = K^T (d x keys) and B = dS^T as [query][key], both read from
            // [key][*] tiles, MN-major; the dS^T columns just read by dK are
            // overwritten only after it (one thread's MMAs run in issue order)
            const uint64_t ka0 = sdesc_sw128(k_addr, 128 * 128, 1024);
            const uint64_t db0 = sdesc_sw128(bo, 128 * 128, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + 128, ka0 + mnmajor_step(kk), db0 + mnmajor_step(kk), kIdQ,
                     kk > 0 ? 1u : 0u);
            mma_commit(&sm.dq_full);
            dq_pending = true;
          }
          if constexpr (!kQ128 && !kQ64) {  // (kQ128: the reducer frees them; kQ64: above)
            mma_commit(&sm.q_empty[qs]);
            mma_commit(&sm.o_empty[qs]);
          }
          if (++qs == kQoStages) { qs = 0; qph ^= 1; }
        }
        if (!ok) break;
        // dK and dV are complete for the epilogue: one commit per item (the
        // grad warps wait for its phase once per item)
        if (x.n_i > 0) mma_commit(&sm.dkv_done);
        mma_commit(&sm.kv_empty);
      }
      if (issued) {
        mma_commit(&sm.final_bar);
        drain_wait(&sm.final_bar, 0, p.wait_ns);
      }
    } else if (kQ64 && warp == 3 && lane == 0) {
      // --------------------------------- dQ issue (fused form, D = 64)
      // A second MMA-issuing thread: at d = 64 one thread cannot issue the
      // 34 products of a step as fast as the tensor pipe runs them.  Per
      // step it issues dK_i and then dQ_i = dS K_j, which reads
      // only dS^T's shared tile (ds_ready, written after the grad warps
      // published P^T and dS^T) and the K_j tile, and writes its own TMEM
      // region (alternately [320,384) and [448,512), once the grad warps
      // have drained dQ_{i-2} from it).  Its products' completion is
      // tracked by its own commits (dk_done, q_empty, dq_done, and kv_empty:
      // K_j's slot is free only when both threads' products of the item are
      // complete).
      constexpr uint32_t kIdQ64 = idesc_bf16_f32(128, 64, 1, 1);  // dQ = dS K
      constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, 1);    // dK += dS^T Q_i
      const uint32_t k_addr = smem_addr(sm.k);
      uint32_t kv_phase = 0, qs = 0, qph = 0, p_phase = 0;
      int64_t n_dq = 0;
      bool issued = false;
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        DkdvPiece pc;
        const DkdvItem x = dkdv_item<kSplit>(p, it, &pc);
        if (kSplit && pc.empty) continue;  // (every role skips the same items)
        if (!mbar_wait(&sm.kv_full, kv_phase, guard)) break;
        kv_phase ^= 1;
        bool ok = true;
        for (int64_t s = 0; s < x.n_i; ++s) {
          // dK_i += dS^T Q_i once the grad warps have published dS^T in TMEM
          // (p_full), while the first thread issues dV_i and the next S^T;
          // that thread waits for dk_done before the next dP^T overwrites
          // the dS^T columns.  Q_i has then been read for the last time.
          if (!mbar_wait(&sm.p_full, p_phase, guard)) { ok = false; break; }
          p_phase ^= 1;
          // (Q_i's load: already complete, as S^T_i has read it)
          if (!mbar_wait(&sm.q_full[qs], qph, guard)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t bq0 = seq_b_base<D, false>(smem_addr(sm.q[qs]));
            const uint32_t acc0 = s > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + 384, tmem + 128 + packed_col(kk), bq0 + seq_b_step<D, false>(kk),
                     kIdG, kk > 0 ? 1u : acc0);
          }
          mma_commit(&sm.dk_done);
          mma_commit(&sm.q_empty[qs]);
          issued = true;
          if (++qs == kQoStages) { qs = 0; qph ^= 1; }
          const int buf = static_cast<int>(n_dq & 1);
          if (n_dq >= 2 &&
              !mbar_wait(&sm.dq_free[buf], static_cast<uint32_t>((n_dq - 2) >> 1) & 1u, guard)) {
            ok = false;
            break;
          }
          // (one barrier per tile: the tile's next write, two steps on, waits
          // for this product through the reducer, so a phase is never missed)
          if (!mbar_wait(&sm.ds_ready[buf], static_cast<uint32_t>(n_dq >> 1) & 1u, guard)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // A = dS^T's [key][query] tile and B = K_j's [key][d] tile, both
          // MN-major
          const uint64_t da0 = sdesc_sw128(smem_addr(sm.ds[buf]), 128 * 128, 1024);
          const uint64_t kb0 = sdesc_sw128(k_addr, 128 * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + (buf ? 448u : 320u), da0 + mnmajor_step(kk), kb0 + mnmajor_step(kk),
                   kIdQ64, kk > 0 ? 1u : 0u);
          mma_commit(&sm.dq_done[buf]);
          ++n_dq;
          issued = true;
        }
        if (!ok) break;
        mma_commit(&sm.kv_empty);
      }
      if (issued) {
        mma_commit(&sm.final_dq);
        drain_wait(&sm.final_dq, 0, p.wait_ns);
      }
    } else if (kQ64 && p.acc_tma && warp == 2 && lane == 0) {
      // ------------------------------------- dQ reducer (fused form, D = 64)
      // Step m: wait for the grad warps' staged scale * dQ_m (fp32, two
      // [128 queries][32 d] boxes with the 128-byte swizzle, in the dS^T
      // tile that dQ_m's product has finished reading), add it into the
      // target with two tensor-map reduce-adds, and free the tile for the
      // dS^T of step m + 2 once the TMA unit has read it.
      uint32_t sf_phase = 0;
      int64_t m = 0;
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        DkdvPiece pc;
        const DkdvItem x = dkdv_item<kSplit>(p, it, &pc);
        if (kSplit && pc.empty) continue;  // (every role skips the same items)
        bool ok = true;
        DkdvCursor cur = kSplit ? dkdv_at(x, pc.s0) : dkdv_first(x);
        for (int64_t s = 0; s < x.n_i; ++s, ++m) {
          int64_t h, i;
          dkdv_take(p, x, cur, h, i);
          if (!mbar_wait(&sm.stage_full, sf_phase, guard)) { ok = false; break; }
          sf_phase ^= 1;
          const uint8_t* src = reinterpret_cast<const uint8_t*>(sm.ds[kQ64 ? (m & 1) : 0]);
          for (int bx = 0; bx < 2; ++bx)
            tma_reduce_add_4d(&tm_acc, src + bx * 16384, 32 * bx, static_cast<int>(i * 128),
                              static_cast<int>(h), static_cast<int>(x.b));
          bulk_commit();
          bulk_wait_read();
          mbar_arrive(&sm.stage_free[m & 1]);
        }
        if (!ok) break;
      }
      bulk_wait_all();
    } else if (kQ128 && warp == 2 && lane == 0) {
      // ------------------------------------------ dQ reducer (fused form)
      // Step by step: wait for the grad warps' staged scale * dQ_i (fp32
      // rows of 128; queries 0..63 in the Q_i slot, 64..127 in the dO_i
      // slot), add it into the accumulator with bulk reduce-adds, and free
      // both slots once the TMA unit has read them.
      uint32_t slot = 0, sf_phase = 0;
      bool any = false;
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        DkdvPiece pc;
        const DkdvItem x = dkdv_item<kSplit>(p, it, &pc);
        if (kSplit && pc.empty) continue;  // (every role skips the same items)
        bool ok = true;
        DkdvCursor cur = kSplit ? dkdv_at(x, pc.s0) : dkdv_first(x);
        for (int64_t s = 0; s < x.n_i; ++s) {
          int64_t h, i;
          dkdv_take(p, x, cur, h, i);
          if (!mbar_wait(&sm.stage_full, sf_phase, guard)) { ok = false; break; }
          sf_phase ^= 1;
          // one bulk group per half: the Q_i slot (queries 0..63) is freed as
          // soon as its group has been read, so that Q_{i+2} loads earlier
          for (int half = 0; half < 2; ++half) {
            const int64_t q0 = i * 128 + 64 * half;
            int64_t rows = p.Lq - q0;
            if (rows > 64) rows = 64;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(half ? sm.d_o[slot] : sm.q[slot]);
            float* dst = p.dq_acc + x.b * p.acc_sb + h * p.acc_sh + q0 * p.acc_sn;
            if (p.acc_tma) {
              // two boxes of [128 d][32 queries] (transposed accumulator)
              for (int bx = 0; bx < 2; ++bx)
                if (q0 + 32 * bx < p.Lq)
                  tma_reduce_add_4d(&tm_acc, src + bx * 16384, static_cast<int>(q0 + 32 * bx), 0,
                                    static_cast<int>(h), static_cast<int>(x.b));
            } else if (rows > 0 && p.acc_sn == 128) {
              bulk_reduce_add_f32(dst, src, static_cast<uint32_t>(rows * 512));
            } else {
              for (int64_t rr = 0; rr < rows; ++rr)
                bulk_reduce_add_f32(dst + rr * p.acc_sn, src + rr * 512, 512u);
            }
            bulk_commit();
          }
          any = true;
          bulk_wait_read_but1();
          mbar_arrive(&sm.q_empty[slot]);
          bulk_wait_read();
          mbar_arrive(&sm.o_empty[slot]);
          if (++slot == kQoStages) slot = 0;
        }
        if (!ok) break;
      }
      if (any) bulk_wait_all();
    }
  } else {
    regs_inc<104>();
    // -------------------------------------------- P^T, dS^T and the epilogue
    const int g = warp - 4;
    const int quad = g & 3, qtr = g >> 2;
    const int row = quad * 32 + lane;  // key row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + 32 * qtr;        // S^T / P^T
    const uint32_t tP = tmem + lane_base + 128 + 32 * qtr;  // dP^T / dS^T
    uint32_t ls = 0, lph = 0, s_phase = 0, dq_phase = 0, gs = 0;
    uint32_t e_count = 0;  // items whose dK / dV have been read out
    const float sl2 = p.scale_log2;
    const float2 sc2 = make_float2(sl2, sl2);
    // D = 64 fused dQ: steps issued so far and the last step's (b, h, i);
    // drain64(m, ...) reads dQ of step m (query row = this lane, 16 of its
    // 64 columns) and frees its TMEM region.  With acc_tma it stages
    // scale * dQ in step m's dS^T tile (which dQ_m's product has finished
    // reading; the next dS^T written there, step m + 2's, waits for the
    // reducer) for the reducer's tensor-map reduce-adds; otherwise it adds
    // scale * dQ into the target with four 16-byte atomics.
    int64_t n_g = 0, pb = 0, ph = 0, pi = 0;
    bool grad_ok = true;
    auto drain64 = [&](int64_t m, int64_t b, int64_t h, int64_t i) -> bool {
      const int buf = static_cast<int>(m & 1);
      if (!mbar_wait(&sm.dq_done[buf], static_cast<uint32_t>(m >> 1) & 1u, guard)) return false;
      tc_fence_after();
      uint32_t w[16];
      tmem_ld16_sync(tmem + lane_base + (buf ? 448u : 320u) + 16 * qtr, w);
      tc_fence_before();
      mbar_arrive(&sm.dq_free[buf]);
      if (p.acc_tma) {
        // box (qtr >> 1) holds d columns [32 (qtr >> 1), +32) as [128
        // queries][32 floats], 128-byte swizzle; four 16-byte stores per
        // thread, conflict-free.  Rows past Lq are clipped by the map.
        const float sc = p.scale;
        uint8_t* line =
            reinterpret_cast<uint8_t*>(sm.ds[kQ64 ? buf : 0]) + (qtr >> 1) * 16384 + row * 128;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const int ch = (qtr & 1) * 4 + c4;  // 16-byte chunk (4 d columns) in the line
          *reinterpret_cast<float4*>(line + ((ch ^ (row & 7)) << 4)) =
              make_float4(__uint_as_float(w[4 * c4]) * sc, __uint_as_float(w[4 * c4 + 1]) * sc,
                          __uint_as_float(w[4 * c4 + 2]) * sc, __uint_as_float(w[4 * c4 + 3]) * sc);
        }
        fence_proxy_async_smem();
        mbar_arrive(&sm.stage_full);
        return true;
      }
      const int64_t qrow = i * 128 + row;
      if (qrow < p.Lq) {
        float* dst = p.dq_acc + b * p.acc_sb + h * p.acc_sh + qrow * p.acc_sn + 16 * qtr;
        const float sc = p.scale;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          red_add_v4_f32(dst + 4 * c4, __uint_as_float(w[4 * c4]) * sc,
                         __uint_as_float(w[4 * c4 + 1]) * sc, __uint_as_float(w[4 * c4 + 2]) * sc,
                         __uint_as_float(w[4 * c4 + 3]) * sc);
      }
      return true;
    };
    for (int64_t r = 0;; ++r) {
      const int64_t it = snake_item(c, r, G);
      if (it >= p.n_items) break;
      DkdvPiece pc;
      const DkdvItem x = dkdv_item<kSplit>(p, it, &pc);
      if (kSplit && pc.empty) continue;  // (every role skips the same items)
      const int64_t key_abs = p.kv_off + x.j * 128 + row;
      bool ok = true;
      DkdvCursor cur = kSplit ? dkdv_at(x, pc.s0) : dkdv_first(x);
      for (int64_t s = 0; s < x.n_i; ++s) {
        int64_t h, i;
        dkdv_take(p, x, cur, h, i);
        // P^T as soon as S^T is in (dP^T may still be in the tensor pipe)
        if (!mbar_wait(&sm.s_ready, s_phase, guard)) { ok = false; break; }
        if (!kRS && !mbar_wait(&sm.lse_full[ls], lph, guard)) { ok = false; break; }
        tc_fence_after();
        // query columns c (of this quarter) with q_off + 128 i + 32 qtr + c
        // >= key_abs are visible
        int cmin = 0;
        if (p.causal) {
          const int64_t tt = key_abs - (p.q_off + i * 128 + 32 * qtr);
          cmin = tt <= 0 ? 0 : (tt > 32 ? 32 : static_cast<int>(tt));
        }
        const float4* l2v = reinterpret_cast<const float4*>(&sm.lse2[ls][32 * qtr]);
        const float4* dlv = reinterpret_cast<const float4*>(&sm.delta[ls][32 * qtr]);
        float pr[32];
        uint32_t pk[16], dk[16];
        {
          uint32_t us[32];
          tmem_ld32(tS, us);
          tmem_ld_wait32(us);
          if constexpr (kRS) {
            // the scores already hold S - LSE/scale; only tiles that straddle
            // the diagonal for this warp need the mask
            const bool need_mask =
                p.causal && p.kv_off + x.j * 128 + quad * 32 + 31 > p.q_off + i * 128 + 32 * qtr;
            if (need_mask)
              p_rows_rs<true>(us, sc2, cmin, pr, pk);
            else
              p_rows_rs<false>(us, sc2, cmin, pr, pk);
          } else {
            p_rows_st(us, sc2, l2v, cmin, pr, pk);
          }
        }
        tmem_st16(tS, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.pt_full);
        // dS^T once dP^T is in
        if (!mbar_wait(&sm.s_full, s_phase, guard)) { ok = false; break; }
        s_phase ^= 1;
        tc_fence_after();
        {
          uint32_t ud[32];
          tmem_ld32(tP, ud);
          tmem_ld_wait32(ud);
          if constexpr (kRS)
            ds_rows_rs(pr, ud, dk);
          else
            ds_rows_st(pr, ud, dlv, dk);
        }
        tmem_st16(tP, dk);
        if constexpr (!kRS) {
          mbar_arrive(&sm.lse_empty[ls]);
          if (++ls == 2) { ls = 0; lph ^= 1; }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full);
        if constexpr (kQ64) {
          // dS^T as bf16 [key][query] (two 64-query boxes, 128-byte swizzle)
          // into its own tile, after P^T and dS^T have been published in
          // TMEM: only dQ_i, which the second MMA thread issues, reads the
          // tile (ds_ready), so these writes stay off the path to dV / dK.
          // The dQ product that last read the tile (two steps back)
          // completed before this warp's previous drain.  With acc_tma the
          // tile has held that step's staged dQ since: wait until the
          // reducer has read it.
          if (p.acc_tma && n_g >= 2 &&
              !mbar_wait(&sm.stage_free[n_g & 1], static_cast<uint32_t>((n_g - 2) >> 1) & 1u,
                         guard)) { ok = false; break; }
          uint8_t* line = reinterpret_cast<uint8_t*>(sm.ds[n_g & 1]) + (qtr >> 1) * 16384 + row * 128;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int ch = (qtr & 1) * 4 + c4;
            *reinterpret_cast<uint4*>(line + ((ch ^ (row & 7)) << 4)) =
                make_uint4(dk[4 * c4], dk[4 * c4 + 1], dk[4 * c4 + 2], dk[4 * c4 + 3]);
          }
          fence_proxy_async_smem();
          mbar_arrive(&sm.ds_ready[n_g & 1]);
          if (n_g >= 1 && !drain64(n_g - 1, pb, ph, pi)) { ok = false; break; }
          pb = x.b; ph = h; pi = i;
          ++n_g;
        }
        if constexpr (kQ128) {
          // dS^T as bf16 [key][query] (two 64-query boxes, 128-byte swizzle,
          // the layout a TMA load of such a tile produces) into the slot of
          // dO_i, once the dV product has finished reading it (the packed
          // pairs stay in registers across the wait: reading them back from
          // TMEM would queue behind the dK product's accesses there)
          if (!mbar_wait(&sm.dv_done, dq_phase, guard)) { ok = false; break; }
          {
            uint8_t* line = reinterpret_cast<uint8_t*>(sm.d_o[gs]) + (qtr >> 1) * 16384 + row * 128;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const int ch = (qtr & 1) * 4 + c4;  // 16-byte chunk (8 queries) in the line
              *reinterpret_cast<uint4*>(line + ((ch ^ (row & 7)) << 4)) =
                  make_uint4(dk[4 * c4], dk[4 * c4 + 1], dk[4 * c4 + 2], dk[4 * c4 + 3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(&sm.ds_full);
          const uint32_t gs_prev = gs;
          if (++gs == 2) gs = 0;
          // dQ_i^T: lane = dimension quad * 32 + lane, columns = this
          // quarter's 32 queries; read it, release the columns, then add
          // scale * dQ^T into the accumulator (one 128-byte row segment per
          // warp instruction)
          if (!mbar_wait(&sm.dq_full, dq_phase, guard)) { ok = false; break; }
          dq_phase ^= 1;
          tc_fence_after();
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + 128 + 32 * qtr, u);
          tmem_ld_wait32(u);
          tc_fence_before();
          mbar_arrive(&sm.dq_drained);
          // stage scale * dQ^T (queries 0..63 in the Q_i slot, 64..127 in
          // the dO_i slot; the dQ^T MMA, complete, was the last reader of
          // both): as [query][d] fp32 rows of 512 bytes (each warp store
          // covers 128 consecutive bytes of one row) or, for the transposed
          // accumulator, as swizzled [d][32 queries] boxes
          if (p.acc_tma) {
            // transposed accumulator: this quarter's 32 queries are box
            // (qtr & 1) of the slot, [128 d][32 queries] with the 128-byte
            // swizzle; eight 16-byte stores per thread, conflict-free
            uint8_t* sb = reinterpret_cast<uint8_t*>(qtr < 2 ? sm.q[gs_prev] : sm.d_o[gs_prev]) +
                          (qtr & 1) * 16384 + row * 128;
            const float sc = p.scale;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<float4*>(sb + ((c ^ (row & 7)) << 4)) =
                  make_float4(__uint_as_float(u[4 * c]) * sc, __uint_as_float(u[4 * c + 1]) * sc,
                              __uint_as_float(u[4 * c + 2]) * sc, __uint_as_float(u[4 * c + 3]) * sc);
          } else {
            float* stage = reinterpret_cast<float*>(qtr < 2 ? sm.q[gs_prev] : sm.d_o[gs_prev]) +
                           (qtr & 1) * 32 * 128 + row;
#pragma unroll
            for (int e = 0; e < 32; ++e) stage[e * 128] = __uint_as_float(u[e]) * p.scale;
          }
          fence_proxy_async_smem();
          mbar_arrive(&sm.stage_full);
        }
      }
      if (!ok) { grad_ok = false; break; }
      // epilogue: half 0 writes dV, half 1 writes dK (times scale)
      if (x.n_i > 0) {
        if (!mbar_wait(&sm.dkv_done, e_count & 1, guard)) { grad_ok = false; break; }
        ++e_count;
        tc_fence_after();
      }
      const int64_t krow = x.j * 128 + row;
      const bool valid = krow < p.Lk;
      // quarters 0, 1: dV columns [0, D/2), [D/2, D); quarters 2, 3: dK
      const uint32_t base_col = (qtr < 2 ? 256u : 384u) + (qtr & 1) * (D / 2);
      const int col0 = (qtr & 1) * (D / 2);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t u[32];
        if (x.n_i > 0) {
          tmem_ld32(tmem + lane_base + base_col + cc * 32, u);
          tmem_ld_wait32(u);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        if (!valid) continue;
        if constexpr (kSplit) {
          // this piece's partial rows, fp32, into its slot
          const int64_t prow = ((pc.piece * p.B + x.b) * p.Hkv + x.hk) * p.Lk + krow;
          store_row32(qtr < 2 ? p.part_dv : p.part_dk, 1, prow * D + col0 + cc * 32, u,
                      qtr < 2 ? 1.f : p.scale, 0);
          continue;
        }
        if (qtr < 2)
          store_row32(p.dv, p.dv_f32,
                      x.b * p.dv_sb + x.hk * p.dv_sh + krow * p.dv_sn + col0 + cc * 32, u, 1.f,
                      p.accumulate);
        else
          store_row32(p.dk, p.dk_f32,
                      x.b * p.dk_sb + x.hk * p.dk_sh + krow * p.dk_sn + col0 + cc * 32, u,
                      p.scale, p.accumulate);
      }
      tc_fence_before();
    }
    if (kQ64 && grad_ok && n_g >= 1) drain64(n_g - 1, pb, ph, pi);  // the last dQ
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

// ======================================================================= dQ
// Query-tile-major.  S = Q K_j^T and dP = dO V_j^T (SS), dS -> bf16 pairs in
// its own TMEM columns, dQ += dS K_j (TS).  The grad warps release the S/dP
// columns as soon as they have loaded them, so the next S/dP products run
// while they compute dS, and dQ(j) runs while dS(j+1) is being computed.
// TMEM: S [0,128), dP [128,256), dQ [256,256+D), dS [384,448).
template <int D, bool kT>
struct DqSmem {
  static constexpr int kStages = 2;
  __nv_bfloat16 q[128 * D];
  __nv_bfloat16 d_o[128 * D];
  __nv_bfloat16 k[kStages][128 * D];
  __nv_bfloat16 v[kStages][128 * D];
  __nv_bfloat16 kt[kT ? 128 * D : 8];
  uint64_t qo_full, qo_empty, final_bar;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t kt_full, kt_empty;
  uint64_t s_full, s_free, p_full, ds_free;
  uint32_t tmem_base;
  int abort;
};

struct DqItem {
  int64_t b, h, hk, i, nkv;
};

__device__ __forceinline__ DqItem dq_item(const BwdParams& p, int64_t it) {
  DqItem x;
  int64_t rank, bh;
  banded_item(it, p.n_qtiles, p.B * p.Hq, &rank, &bh);
  x.i = p.n_qtiles - 1 - rank;  // the longest key range first
  x.b = bh / p.Hq;
  x.h = bh % p.Hq;
  x.hk = x.h / (p.Hq / p.Hkv);
  x.nkv = p.row_list == nullptr ? fwd_kv_tiles(x.i, p.Lq, p.Lk, p.q_off, p.kv_off, p.causal)
                                 : p.row_count[x.i];
  return x;
}

// Key tile at position j of a dQ item.
__device__ __forceinline__ int64_t dq_key_tile(const BwdParams& p, const DqItem& x, int64_t j) {
  return p.row_list == nullptr ? j : p.row_list[x.i * p.n_ktiles + j];
}

template <int D, bool kT>
__global__ void __launch_bounds__(640, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_kt, const BwdParams p) {
  using Sm = DqSmem<D, kT>;
  constexpr int kStages = Sm::kStages;
  constexpr int kTile = 128 * D * 2;
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
    mbar_init(&sm.kt_full, 1);
    mbar_init(&sm.kt_empty, 1);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, 512);
    mbar_init(&sm.p_full, 512);
    mbar_init(&sm.ds_free, 1);
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
  if (p.trace != nullptr && threadIdx.x == 0)
    trace_begin(p.trace, p.trace_kid, p.n_items, global_timer_ns());

  // 640 threads launched at <= 96 registers (61,440): the load/MMA
  // warpgroup keeps 64, the four grad warpgroups take 104:
  // 128 * 64 + 512 * 104 = 61,440 <= 61,440.
  if (warp < 4) {
    regs_dec<64>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------- loads: Q, dO and K/V ring
      uint32_t stage = 0, phase = 0, qo_phase = 0;
      int64_t r = 0;
      for (;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        const DqItem x = dq_item(p, it);
        if (x.nkv == 0) continue;
        if (!mbar_wait(&sm.qo_empty, qo_phase ^ 1, guard)) break;
        qo_phase ^= 1;
        mbar_arrive_expect_tx(&sm.qo_full, 2 * kTile);
        load_tile<D, false>(sm.q, &tm_q, &sm.qo_full, x.i * 128, x.h, x.b);
        load_tile<D, false>(sm.d_o, &tm_do, &sm.qo_full, x.i * 128, x.h, x.b);
        bool ok = true;
        for (int64_t j = 0; j < x.nkv; ++j) {
          if (!mbar_wait(&sm.kv_empty[stage], phase ^ 1, guard)) { ok = false; break; }
          mbar_arrive_expect_tx(&sm.kv_full[stage], 2 * kTile);
          const int64_t kt = dq_key_tile(p, x, j);
          load_tile<D, false>(sm.k[stage], &tm_k, &sm.kv_full[stage], kt * 128, x.hk, x.b);
          load_tile<D, false>(sm.v[stage], &tm_v, &sm.kv_full[stage], kt * 128, x.hk, x.b);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
      if (p.trace != nullptr) trace_items(p.trace, r);
    } else if (kT && warp == 0 && lane == 1) {
      // ------------------------- loads: K^T ring (its own thread, so that a
      // K^T slot still in use never holds back the K/V prefetch)
      uint32_t kt_phase = 0;
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        const DqItem x = dq_item(p, it);
        bool ok = true;
        for (int64_t j = 0; j < x.nkv; ++j) {
          if (!mbar_wait(&sm.kt_empty, kt_phase ^ 1, guard)) { ok = false; break; }
          kt_phase ^= 1;
          mbar_arrive_expect_tx(&sm.kt_full, kTile);
          load_tile<D, true>(sm.kt, &tm_kt, &sm.kt_full, dq_key_tile(p, x, j) * 128, x.hk,
                             x.b);
        }
        if (!ok) break;
      }
    } else if (warp == 1 && lane == 0) {
      // ----------------------------------------------------------- MMA issue
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, kT ? 0 : 1);
      uint32_t kst = 0, kph = 0, kt_phase = 0, qo_phase = 0, sf_phase = 0, pf_phase = 0;
      bool s_outstanding = false, issued = false;
      const uint32_t q_addr = smem_addr(sm.q), o_addr = smem_addr(sm.d_o);
      for (int64_t r = 0;; ++r) {
        const int64_t it = snake_item(c, r, G);
        if (it >= p.n_items) break;
        const DqItem x = dq_item(p, it);
        if (x.nkv == 0) continue;
        if (!mbar_wait(&sm.qo_full, qo_phase, guard)) break;
        qo_phase ^= 1;
        tc_fence_after();
        bool ok = true;
        uint32_t prev = 0;
        for (int64_t j = 0; j <= x.nkv; ++j) {
          const uint32_t cur = kst;
          if (j < x.nkv) {
            if (!mbar_wait(&sm.kv_full[kst], kph, guard)) { ok = false; break; }
            if (s_outstanding) {  // the grad warps have loaded the last S/dP
              if (!mbar_wait(&sm.s_free, sf_phase, guard)) { ok = false; break; }
              sf_phase ^= 1;
            }
            tc_fence_after();
            mma_rows_by_rows<D>(tmem + 0, q_addr, smem_addr(sm.k[kst]), kIdS);
            mma_rows_by_rows<D>(tmem + 128, o_addr, smem_addr(sm.v[kst]), kIdS);
            mma_commit(&sm.s_full);
            s_outstanding = true;
            issued = true;
            if constexpr (kT) mma_commit(&sm.kv_empty[kst]);  // K_j, V_j done
            if (++kst == kStages) { kst = 0; kph ^= 1; }
          }
          if (j > 0) {  // dQ += dS(j-1) K_{j-1}
            if (!mbar_wait(&sm.p_full, pf_phase, guard)) { ok = false; break; }
            pf_phase ^= 1;
            uint64_t b0;
            if constexpr (kT) {
              if (!mbar_wait(&sm.kt_full, kt_phase, guard)) { ok = false; break; }
              kt_phase ^= 1;
              b0 = sdesc_sw128(smem_addr(sm.kt), 16, 1024);
            } else {
              b0 = sdesc_sw128(smem_addr(sm.k[prev]), 128 * 128, 1024);
            }
            tc_fence_after();
            const uint32_t acc0 = j > 1 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + 256, tmem + 384 + kk * 8,
                     b0 + (kT ? kmajor_step(kk, D) : mnmajor_step(kk)), kIdG,
                     kk > 0 ? 1u : acc0);
            mma_commit(&sm.ds_free);
            if constexpr (kT) mma_commit(&sm.kt_empty);
            else mma_commit(&sm.kv_empty[prev]);
          }
          prev = cur;
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
    regs_inc<104>();
    // ------------------------------------------------------ dS and epilogue
    const int g = warp - 4;
    const int quad = g & 3, qtr = g >> 2;
    const int row = quad * 32 + lane;  // query row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_base + 32 * qtr;
    const uint32_t tP = tmem + lane_base + 128 + 32 * qtr;
    const uint32_t tD = tmem + lane_base + 384 + 16 * qtr;  // packed dS of this quarter
    uint32_t s_phase = 0, n_ds = 0;
    const float sl2 = p.scale_log2;
    const float2 sc2 = make_float2(sl2, sl2);
    for (int64_t r = 0;; ++r) {
      const int64_t it = snake_item(c, r, G);
      if (it >= p.n_items) break;
      const DqItem x = dq_item(p, it);
      const int64_t qrow = x.i * 128 + row;
      const bool valid = qrow < p.Lq;
      if (x.nkv == 0) {  // no visible key: dQ = 0 (or unchanged when accumulating)
        if (valid && !p.accumulate && 32 * qtr < D) {
          uint32_t z[32] = {};
          store_row32(p.dq, p.dq_f32, x.b * p.dq_sb + x.h * p.dq_sh + qrow * p.dq_sn + 32 * qtr,
                      z, 0.f, 0);
        }
        continue;
      }
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
        uint32_t us[32], ud[32];
        ld_two(tS, tP, us, ud);
        tc_fence_before();
        mbar_arrive(&sm.s_free);  // S/dP columns may be overwritten now
        // visible key columns of this quarter: c <= climit
        const int64_t kb = dq_key_tile(p, x, j) * 128 + 32 * qtr;
        int64_t lim = 31;
        if (kb + 32 > p.Lk) lim = p.Lk - kb - 1;
        if (p.causal) {
          const int64_t c2 = p.q_off + qrow - p.kv_off - kb;
          if (c2 < lim) lim = c2;
        }
        const int climit = lim < -1 ? -1 : static_cast<int>(lim);
        // every column visible to every row of this warp: no mask needed
        const bool need_mask =
            kb + 32 > p.Lk ||
            (p.causal && p.q_off + x.i * 128 + quad * 32 - p.kv_off - kb < 31);
        uint32_t dk[16];
        if (need_mask)
          grad_cols_dq<true>(us, ud, sc2, nl, nd, climit, dk);
        else
          grad_cols_dq<false>(us, ud, sc2, nl, nd, climit, dk);
        // the dS columns are free once the previous dQ product has read them
        if (n_ds > 0) {
          if (!mbar_wait(&sm.ds_free, (n_ds - 1) & 1, guard)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st16(tD, dk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.p_full);
        ++n_ds;
      }
      if (!ok) break;
      if (!mbar_wait(&sm.ds_free, (n_ds - 1) & 1, guard)) break;
      tc_fence_after();
      // epilogue: quarter q writes dQ columns [32 q, 32 q + 32) (times scale)
      if (32 * qtr < D) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + 256 + 32 * qtr, u);
        tmem_ld_wait32(u);
        if (valid)
          store_row32(p.dq, p.dq_f32,
                      x.b * p.dq_sb + x.h * p.dq_sh + qrow * p.dq_sn + 32 * qtr, u, p.scale,
                      p.accumulate);
      }
      tc_fence_before();
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

// dq (bf16 or f32 view) = acc (dense fp32 [B*Hq*Lq][D]), optionally added
// to what dq holds; four columns per thread (c4 = D / 4 per row).
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, void* dq,
                                                         int f32, int64_t sb, int64_t sh,
                                                         int64_t sn, int64_t Hq, int64_t Lq,
                                                         int64_t total4, int c4, int accumulate) {
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total4;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t rowi = t / c4;
    const int64_t col = (t % c4) * 4;
    const int64_t n = rowi % Lq, bh = rowi / Lq;
    const int64_t off = (bh / Hq) * sb + (bh % Hq) * sh + n * sn + col;
    float4 a = reinterpret_cast<const float4*>(acc)[t];
    if (f32) {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(dq) + off);
      if (accumulate) {
        const float4 o = *d;
        a.x += o.x; a.y += o.y; a.z += o.z; a.w += o.w;
      }
      *d = a;
    } else {
      uint2* d = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(dq) + off);
      if (accumulate) {
        const uint2 o = *d;
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&o.x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&o.y);
        a.x += __low2float(lo); a.y += __high2float(lo);
        a.z += __low2float(hi); a.w += __high2float(hi);
      }
      *d = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
    }
  }
}

// dq (bf16 or f32 view, D = 128) = the transposed accumulator
// [B*Hq][128][Np], optionally added to what dq holds.  A block moves 32
// queries x 128 dims through shared memory: reads along queries, writes
// along d (four columns per thread).
__global__ void __launch_bounds__(256) dq_convert_t_kernel(const float* __restrict__ acc, void* dq,
                                                           int f32, int64_t sb, int64_t sh,
                                                           int64_t sn, int64_t Hq, int64_t Lq,
                                                           int64_t np, int accumulate) {
  __shared__ float tile[128][33];
  const int64_t bh = blockIdx.y;
  const int64_t q0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const float* src = acc + bh * 128 * np;
  for (int d = w; d < 128; d += 8)
    tile[d][lane] = (q0 + lane < Lq) ? src[d * np + q0 + lane] : 0.f;
  __syncthreads();
  const int64_t b = bh / Hq, h = bh % Hq;
  // lane l writes dimensions (2l, 2l+1) and (64+2l, 65+2l) of each query:
  // the tile reads of a warp then fall on 16 distinct banks twice (a
  // two-way conflict), where four consecutive dimensions per lane gave four
  // reads of four ways each
  for (int qq = w; qq < 32; qq += 8) {
    const int64_t q = q0 + qq;
    if (q >= Lq) break;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int d0 = 64 * half + 2 * lane;
      float2 a = make_float2(tile[d0][qq], tile[d0 + 1][qq]);
      const int64_t off = b * sb + h * sh + q * sn + d0;
      if (f32) {
        float2* d = reinterpret_cast<float2*>(static_cast<float*>(dq) + off);
        if (accumulate) {
          const float2 o = *d;
          a.x += o.x; a.y += o.y;
        }
        *d = a;
      } else {
        uint32_t* d = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(dq) + off);
        if (accumulate) {
          const uint32_t o = *d;
          const __nv_bfloat162 pr = *reinterpret_cast<const __nv_bfloat162*>(&o);
          a.x += __low2float(pr); a.y += __high2float(pr);
        }
        *d = pack_bf16(a.x, a.y);
      }
    }
  }
}

bool map_rows(CUtensorMap* m, const lsx_tensor& t) {
  return make_map_bf16_4d(m, t.data, t.B, t.H, t.N, t.D, t.stride_b, t.stride_h, t.stride_n,
                          128);
}

// map over a transposed copy [B, H, D, Np] of t (boxes of 64 positions x D rows)
bool map_transposed(CUtensorMap* m, const lsx_tensor& t, void* copy, int box_rows) {
  const int64_t np = transposed_row_len(t.N);
  return make_map_bf16_4d(m, copy, t.B, t.H, t.D, t.N, t.H * t.D * np, t.D * np, np, box_rows);
}

bool map_ones(CUtensorMap* m, void* ones) {
  return make_map_bf16_rows8(m, ones, 1, 1, 256);
}

// The pieces of split key columns (BwdSplit): one warp per key row of dK
// and dV, lane l owning columns [l E, l E + E).  A row has as many pieces as
// its item has: ceil(steps / piece_w), steps = the query tiles that see its
// key tile times the heads of the group (from the same causal geometry the
// kernel used); pieces are summed in the order 0, 1, ...
template <int D>
__global__ void __launch_bounds__(256) dkdv_sum_pieces_kernel(const BwdParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t rows = p.B * p.Hkv * p.Lk;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = w0; row < rows; row += nw) {
    const int64_t n = row % p.Lk, bh = row / p.Lk;
    const int64_t b = bh / p.Hkv, hk = bh % p.Hkv;
    const int64_t steps = (p.n_qtiles - q_tile_begin(p, n / 128)) * (p.Hq / p.Hkv);
    const int64_t parts = (steps + p.piece_w - 1) / p.piece_w;
    float ak[E], av[E];
#pragma unroll
    for (int e = 0; e < E; ++e) ak[e] = av[e] = 0.f;
    for (int64_t q = 0; q < parts; ++q) {
      const int64_t off = (q * rows + row) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        ak[e] += __ldcs(p.part_dk + off + e);
        av[e] += __ldcs(p.part_dv + off + e);
      }
    }
    const int64_t ok = b * p.dk_sb + hk * p.dk_sh + n * p.dk_sn + lane * E;
    const int64_t ov = b * p.dv_sb + hk * p.dv_sh + n * p.dv_sn + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (p.dk_f32)
        static_cast<float*>(p.dk)[ok + e] = ak[e];
      else
        static_cast<__nv_bfloat16*>(p.dk)[ok + e] = __float2bfloat16_rn(ak[e]);
      if (p.dv_f32)
        static_cast<float*>(p.dv)[ov + e] = av[e];
      else
        static_cast<__nv_bfloat16*>(p.dv)[ov + e] = __float2bfloat16_rn(av[e]);
    }
  }
}

template <int D>
int launch_bwd_tc_d(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                    const lsx_tensor& lse, const lsx_tensor& d_o, const float* delta,
                    const BwdCopies& cp, int64_t q_off, int64_t kv_off, int causal,
                    float scale, const lsx_tensor& dq, const lsx_tensor& dk,
                    const lsx_tensor& dv, int accumulate, const DeviceCtx& ctx,
                    cudaStream_t s, const BlockLists* bl, const BwdSplit* split) {
  // fused dK/dV/dQ: D = 128, not in deterministic mode, and somewhere to
  // add dQ into (the fp32 accumulator in the workspace, or an f32 dq)
  const bool fused = !ctx.deterministic && (cp.dq_acc != nullptr || dq.dtype == LSX_F32);
  // add straight into an f32 dq when its rows are contiguous (one bulk add
  // per half tile) or when there is no accumulator; a strided dq with the
  // workspace goes through the accumulator (row-by-row adds are 2x slower)
  const bool direct = fused && dq.dtype == LSX_F32 && (dq.stride_n == D || cp.dq_acc == nullptr);
  const bool tr = !fused && cp.kt != nullptr;
  const bool rs = cp.stats.rows != nullptr;
  CUtensorMap tq, tk, tv, tdo, tkt, trs, tones;
  if (!map_rows(&tq, q) || !map_rows(&tk, k) || !map_rows(&tv, v) || !map_rows(&tdo, d_o))
    return LSX_ERR_LAUNCH;
  if (tr) {
    const int rc = launch_transpose(k, cp.kt, s);
    if (rc != LSX_OK) return rc;
    if (!map_transposed(&tkt, k, cp.kt, D)) return LSX_ERR_LAUNCH;
  } else {
    tkt = tk;
  }
  if (rs) {
    if (!make_map_bf16_rows8(&trs, cp.stats.rows, q.B, q.H, q.N) ||
        !map_ones(&tones, cp.stats.ones))
      return LSX_ERR_LAUNCH;
  } else {
    trs = tk;
    tones = tk;
  }
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
  p.row_count = bl ? bl->row_count : nullptr;
  p.row_list = bl ? bl->row_list : nullptr;
  p.col_count = bl ? bl->col_count : nullptr;
  p.col_list = bl ? bl->col_list : nullptr;
  p.dq_acc = nullptr;
  p.acc_sb = p.acc_sh = p.acc_sn = 0;
  p.trace = nullptr;
  p.trace_kid = 0;
  p.piece_w = 0;
  p.kmax = 1;
  p.part_dk = p.part_dv = nullptr;
  const bool split_on = split != nullptr && split->piece_w > 0;
  if (split_on) {
    // the fused form with the statistics on the tensor cores only
    if (!fused || !rs || bl != nullptr || accumulate || split->kmax < 1)
      return LSX_ERR_UNSUPPORTED;
    p.piece_w = split->piece_w;
    p.kmax = split->kmax;
    p.part_dk = split->part_dk;
    p.part_dv = split->part_dv;
  }

  // dK, dV (and dQ): items (key tile, b, kv head), times the pieces if split
  p.n_items = p.n_ktiles * q.B * k.H * p.kmax;
  CUtensorMap tacc = tk;  // (unused unless p.acc_tma)
  p.acc_tma = 0;
  if (fused) {
    if (direct) {
      p.dq_acc = static_cast<float*>(dq.data);
      p.acc_sb = dq.stride_b; p.acc_sh = dq.stride_h; p.acc_sn = dq.stride_n;
      if (!accumulate) {
        const int rc = launch_zero(dq, ctx, s);
        if (rc != LSX_OK) return rc;
      }
    } else if (D == 128) {
      // transposed accumulator [B][Hq][128][Np], added into by tensor-map
      // reduce-adds of [128 d][32 queries] boxes
      const int64_t np = dq_acc_pitch(q.N);
      p.dq_acc = cp.dq_acc;
      p.acc_tma = 1;
      p.acc_sn = 1; p.acc_sh = 128 * np; p.acc_sb = q.H * 128 * np;
      if (!make_map_f32_rows32(&tacc, cp.dq_acc, q.B, q.H, 128, q.N, np)) return LSX_ERR_LAUNCH;
      if (cudaMemsetAsync(cp.dq_acc, 0, static_cast<size_t>(q.B * q.H * 128 * np) * sizeof(float),
                          s) != cudaSuccess)
        return LSX_ERR_LAUNCH;
    } else {
      p.dq_acc = cp.dq_acc;
      p.acc_sn = D; p.acc_sh = q.N * D; p.acc_sb = q.H * q.N * D;
      if (cudaMemsetAsync(cp.dq_acc, 0, static_cast<size_t>(q.B * q.H * q.N * D) * sizeof(float),
                          s) != cudaSuccess)
        return LSX_ERR_LAUNCH;
    }
    // D = 64: staged [128 queries][32 d] boxes added through a tensor map
    // when the target allows one (else 16-byte atomics from registers)
    if (D == 64 && make_map_f32_box32x128(&tacc, p.dq_acc, q.B, q.H, q.N, D, p.acc_sb, p.acc_sh,
                                          p.acc_sn))
      p.acc_tma = 1;
    const size_t smem = sizeof(DkdvSmem<D>) + 1024;
    auto kern = split_on ? dkdv_kernel<D, true, true, true>
                         : (rs ? dkdv_kernel<D, true, true> : dkdv_kernel<D, false, true>);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LSX_ERR_LAUNCH;
    const int64_t grid = p.n_items < ctx.sm_count ? p.n_items : ctx.sm_count;
    p.trace_kid = kKidBwdFused;
    p.trace = trace_record(kKidBwdFused, grid);
    timing_begin(kKidBwdFused, s);
    kern<<<static_cast<unsigned>(grid), 640, smem, s>>>(tq, tk, tv, tdo, trs, tones, tacc, p);
    timing_end(kKidBwdFused, s);
    if (cudaGetLastError() != cudaSuccess) return LSX_ERR_LAUNCH;
    if (split_on) {
      const int64_t rows = k.B * k.H * k.N;
      int64_t blocks = (rows * 32 + 255) / 256;
      if (blocks > 8 * ctx.sm_count) blocks = 8 * ctx.sm_count;
      timing_begin(kKidTreeMerge, s);
      dkdv_sum_pieces_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, s>>>(p);
      timing_end(kKidTreeMerge, s);
      if (cudaGetLastError() != cudaSuccess) return LSX_ERR_LAUNCH;
    }
    if (direct) return LSX_OK;
    if (D == 128) {
      timing_begin(kKidDqConvert, s);
      const dim3 cgrid(static_cast<unsigned>(ceil_div(q.N, 32)), static_cast<unsigned>(q.B * q.H));
      dq_convert_t_kernel<<<cgrid, 256, 0, s>>>(cp.dq_acc, dq.data, dq.dtype == LSX_F32,
                                                dq.stride_b, dq.stride_h, dq.stride_n, q.H, q.N,
                                                dq_acc_pitch(q.N), accumulate);
      timing_end(kKidDqConvert, s);
      return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
    }
    const int64_t total4 = q.B * q.H * q.N * (D / 4);
    int64_t blocks = (total4 + 255) / 256;
    if (blocks > 8 * ctx.sm_count) blocks = 8 * ctx.sm_count;
    timing_begin(kKidDqConvert, s);
    dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        cp.dq_acc, dq.data, dq.dtype == LSX_F32, dq.stride_b, dq.stride_h, dq.stride_n, q.H, q.N,
        total4, D / 4, accumulate);
    timing_end(kKidDqConvert, s);
    return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
  }
  {
    const size_t smem = sizeof(DkdvSmem<D>) + 1024;
    auto kern = rs ? dkdv_kernel<D, true, false> : dkdv_kernel<D, false, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LSX_ERR_LAUNCH;
    const int64_t grid = p.n_items < ctx.sm_count ? p.n_items : ctx.sm_count;
    p.trace_kid = kKidDkdv;
    p.trace = trace_record(kKidDkdv, grid);
    timing_begin(kKidDkdv, s);
    kern<<<static_cast<unsigned>(grid), 640, smem, s>>>(tq, tk, tv, tdo, trs, tones, tk, p);
    timing_end(kKidDkdv, s);
    if (cudaGetLastError() != cudaSuccess) return LSX_ERR_LAUNCH;
  }
  // dQ: items (query tile, b, head)
  p.n_items = p.n_qtiles * q.B * q.H;
  {
    const size_t smem = (tr ? sizeof(DqSmem<D, true>) : sizeof(DqSmem<D, false>)) + 1024;
    auto kern = tr ? dq_kernel<D, true> : dq_kernel<D, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return LSX_ERR_LAUNCH;
    const int64_t grid = p.n_items < ctx.sm_count ? p.n_items : ctx.sm_count;
    p.trace_kid = kKidDq;
    p.trace = trace_record(kKidDq, grid);
    timing_begin(kKidDq, s);
    kern<<<static_cast<unsigned>(grid), 640, smem, s>>>(tq, tk, tv, tdo, tkt, p);
    timing_end(kKidDq, s);
    if (cudaGetLastError() != cudaSuccess) return LSX_ERR_LAUNCH;
  }
  return LSX_OK;
}

}  // namespace

// Scratch behind delta: [selector tiles, 4 KiB][row statistics, 16 bytes
// per query row][one region holding either the fp32 dQ accumulator (D = 128)
// or the key-contiguous copy of K].
namespace {
size_t stats_bytes(const lsx_tensor& q) {
  const size_t rows = static_cast<size_t>(q.B * q.H * q.N);
  return (2 * 128 * 16 + rows * 16 + 255) / 256 * 256;
}
size_t scratch_bytes(const lsx_tensor& q, const lsx_tensor& k) {
  size_t n = transposed_bytes(k);
  // the D = 128 accumulator is transposed with rows padded to dq_acc_pitch
  const int64_t rows = q.D == 128 ? dq_acc_pitch(q.N) : q.N;
  const size_t acc = static_cast<size_t>(q.B * q.H * rows * q.D) * sizeof(float);
  if (acc > n) n = acc;
  return (n + 255) / 256 * 256;
}
}  // namespace

size_t bwd_tc_copies_bytes(const lsx_tensor& q, const lsx_tensor& k) {
  return stats_bytes(q) + scratch_bytes(q, k);
}

BwdCopies bwd_tc_copies(const lsx_tensor& q, const lsx_tensor& k, void* base) {
  (void)k;
  BwdCopies c;
  char* st = static_cast<char*>(base);
  c.stats.ones = st;
  c.stats.rows = st + 2 * 128 * 16;
  char* scratch = st + stats_bytes(q);
  c.kt = scratch;
  c.dq_acc = reinterpret_cast<float*>(scratch);
  return c;
}

int launch_bwd_tc(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                  const lsx_tensor& lse, const lsx_tensor& d_o, const float* delta,
                  const BwdCopies& cp, int64_t q_off, int64_t kv_off, int causal,
                  float scale, const lsx_tensor& dq, const lsx_tensor& dk,
                  const lsx_tensor& dv, int accumulate, const DeviceCtx& ctx,
                  cudaStream_t s, const BlockLists* bl) {
  if (q.D == 128)
    return launch_bwd_tc_d<128>(q, k, v, lse, d_o, delta, cp, q_off, kv_off, causal, scale, dq,
                                dk, dv, accumulate, ctx, s, bl, nullptr);
  if (q.D == 64)
    return launch_bwd_tc_d<64>(q, k, v, lse, d_o, delta, cp, q_off, kv_off, causal, scale, dq,
                               dk, dv, accumulate, ctx, s, bl, nullptr);
  return LSX_ERR_UNSUPPORTED;
}

int launch_bwd_tc_split(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                        const lsx_tensor& lse, const lsx_tensor& d_o, const float* delta,
                        const BwdCopies& cp, int64_t q_off, int64_t kv_off, int causal,
                        float scale, const lsx_tensor& dq, const lsx_tensor& dk,
                        const lsx_tensor& dv, const BwdSplit& split, const DeviceCtx& ctx,
                        cudaStream_t s) {
  if (split.piece_w <= 0) return LSX_ERR_UNSUPPORTED;
  if (q.D == 128)
    return launch_bwd_tc_d<128>(q, k, v, lse, d_o, delta, cp, q_off, kv_off, causal, scale, dq,
                                dk, dv, 0, ctx, s, nullptr, &split);
  if (q.D == 64)
    return launch_bwd_tc_d<64>(q, k, v, lse, d_o, delta, cp, q_off, kv_off, causal, scale, dq,
                               dk, dv, 0, ctx, s, nullptr, &split);
  return LSX_ERR_UNSUPPORTED;
}

}  // namespace lsx
