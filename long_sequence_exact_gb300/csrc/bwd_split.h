// bwd_split.h -- the fused backward with key columns split into pieces (few
// heads, long rows) and the sum of the pieces.
#pragma once

#include "internal.h"

namespace lsx {

// Each dK/dV item's steps (query tiles of the heads of its group) are cut
// into pieces of piece_w steps; piece i of every item writes its partial
// dK, dV (fp32; dK already times scale) to slot i of part_dk, part_dv
// [kmax][B][Hkv][Lk][D]; the partials are then summed row by row into dk,
// dv.  dQ is added into its accumulator by every piece as in the unsplit
// kernel.
struct BwdSplit {
  int64_t piece_w = 0;  // steps per piece
  int64_t kmax = 0;     // pieces of the longest item
  float* part_dk = nullptr;
  float* part_dv = nullptr;
};

// launch_bwd_tc's fused form (full workspace copies, no block lists, no
// accumulation) with the split above.
int launch_bwd_tc_split(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                        const lsx_tensor& lse, const lsx_tensor& d_o, const float* delta,
                        const BwdCopies& cp, int64_t q_off, int64_t kv_off, int causal,
                        float scale, const lsx_tensor& dq, const lsx_tensor& dk,
                        const lsx_tensor& dv, const BwdSplit& split, const DeviceCtx& ctx,
                        cudaStream_t s);

}  // namespace lsx
