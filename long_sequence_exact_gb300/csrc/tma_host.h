// tma_host.h -- host-side construction of TMA tensor maps for [B, H, N, D]
// bf16 views (D contiguous).  The driver entry point is fetched through the
// runtime so the library does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace lsx {

// The driver's encoder, looked up on first use (again after a failed look-up)
// and cached; callers on several threads may get here at the same time.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_acquire);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      cached.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// Tiled map over a bf16 tensor with dims (innermost first) {D, N, H, B} and
// element strides {1, sn, sh, sb}.  Box = {64, box_rows, 1, 1} with the
// 128-byte swizzle, so one box is box_rows rows of 128 bytes, matching the
// K-major / MN-major SW128 shared-memory layouts the MMAs read (or, with
// swizzle = false, plain row-major [box_rows][64]).  Rows beyond N read as
// zero.  Returns false when the driver rejects the map.
inline bool make_map_bf16_4d(CUtensorMap* map, const void* base, int64_t B,
                             int64_t H, int64_t N, int64_t D, int64_t sb,
                             int64_t sh, int64_t sn, uint32_t box_rows,
                             bool swizzle = true) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  // a stride of an extent-1 dimension is never used; give it a legal value
  const int64_t esz = 2;
  if (H == 1) sh = N * sn;
  if (B == 1) sb = H * sh;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)H,
                        (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)(sn * esz), (cuuint64_t)(sh * esz),
                           (cuuint64_t)(sb * esz)};
  cuuint32_t box[4] = {64u, box_rows, 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled map over a dense bf16 array [B][H][N][8] (16 bytes per row), box
// {8, 128, 1, 1} without swizzle: one box is 128 rows of 16 bytes, i.e. 16
// consecutive 8 x 16-byte core matrices.  Rows beyond N read as zero.
inline bool make_map_bf16_rows8(CUtensorMap* map, const void* base, int64_t B,
                                int64_t H, int64_t N) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {8u, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {16u, (cuuint64_t)(N * 16), (cuuint64_t)(H * N * 16)};
  cuuint32_t box[4] = {8u, 128u, 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled map over a dense fp32 array [B][H][R][Np] (Np = row pitch in
// elements, a multiple of 4; the first N elements of each row are the
// tensor), box {32, R, 1, 1} with the 128-byte swizzle: one box is R rows of
// 32 floats.  Used as the destination of bulk reduce-adds; elements past N
// are not touched.  Returns false when the driver rejects the map.
inline bool make_map_f32_rows32(CUtensorMap* map, const void* base, int64_t B, int64_t H,
                                int64_t R, int64_t N, int64_t Np) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[4] = {(cuuint64_t)N, (cuuint64_t)R, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)(Np * 4), (cuuint64_t)(R * Np * 4),
                           (cuuint64_t)(H * R * Np * 4)};
  cuuint32_t box[4] = {32u, (cuuint32_t)R, 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tiled map over an fp32 tensor with dims (innermost first) {D, N, H, B} and
// element strides {1, sn, sh, sb}, box {32, 128, 1, 1} with the 128-byte
// swizzle: one box is 128 rows of 32 floats.  Used as the destination of
// tensor-map reduce-adds; rows past N are not touched.  Returns false when
// the base is not 16-byte aligned, a stride is not a multiple of 16 bytes or
// the driver rejects the map (the caller then adds another way).
inline bool make_map_f32_box32x128(CUtensorMap* map, const void* base, int64_t B, int64_t H,
                                   int64_t N, int64_t D, int64_t sb, int64_t sh, int64_t sn) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr || B <= 0 || H <= 0 || N <= 0 || D < 32) return false;
  if (H == 1) sh = N * sn;  // strides of extent-1 dimensions are never used
  if (B == 1) sb = H * sh;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || sn <= 0 || sh <= 0 || sb <= 0 ||
      (sn * 4) % 16 != 0 || (sh * 4) % 16 != 0 || (sb * 4) % 16 != 0)
    return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)(sn * 4), (cuuint64_t)(sh * 4), (cuuint64_t)(sb * 4)};
  cuuint32_t box[4] = {32u, 128u, 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace lsx
