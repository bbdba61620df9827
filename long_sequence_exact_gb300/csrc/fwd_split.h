// fwd_split.h -- the forward with rows split into key pieces (few heads,
// long rows) and the merge of the pieces.
#pragma once

#include "internal.h"

namespace lsx {

// Each query pair's visible key tiles are cut into pieces of piece_w tiles;
// piece i of every pair writes its normalised partial (fp32 O, LSE) to slot
// i of part_o [kmax][B][Hq][Lq][D] and part_lse [kmax][B][Hq][Lq], which
// launch_merge_pieces then combines row by row.
struct FwdSplit {
  int64_t piece_w = 0;  // key tiles per piece
  int64_t kmax = 0;     // pieces of the longest pair
  float* part_o = nullptr;
  float* part_lse = nullptr;
};

// The forward of launch_fwd_tc (no block lists, no accumulation) with its
// rows split as `split` says.
int launch_fwd_tc_split(const lsx_tensor& q, const lsx_tensor& k, const lsx_tensor& v,
                        int64_t q_off, int64_t kv_off, int causal, float scale,
                        const lsx_tensor& o, const lsx_tensor& lse, void* vt,
                        const FwdSplit& split, const DeviceCtx& ctx, cudaStream_t s);

// The LSE-weighted merge of each row's pieces (as many as its query pair has:
// ceil(visible key tiles / piece_w)) into o (bf16 or f32) and lse.
int launch_merge_pieces(const FwdSplit& split, int64_t q_off, int64_t kv_off, int causal,
                        int64_t Lk, const lsx_tensor& o, const lsx_tensor& lse,
                        const DeviceCtx& ctx, cudaStream_t s);

}  // namespace lsx
