// layout.cu -- transposed copies of bf16 [B, H, N, D] views, written as dense
// [B, H, D, Np] (Np = N rounded up to 8 so every row starts 16-byte aligned).
//
// The tensor cores read an operand fastest when its reduction dimension is
// contiguous in shared memory ("K-major").  The P.V product of the forward
// and the dV, dK, dQ products of the backward reduce over the sequence axis,
// while V, dO, Q and K are stored with d contiguous; feeding them as they are
// makes the MMA read a transposed ("MN-major") operand, which measured about
// 2.2x slower per instruction.  One bandwidth-bound pass writes the
// sequence-contiguous copy instead (read + write of the tensor once).
#include <cuda_bf16.h>

#include "internal.h"

namespace lsx {
namespace {

// One 64 (n) x 64 (d) tile per block of 256 threads, staged in shared memory.
__global__ void __launch_bounds__(256) transpose_kernel(lsx_tensor in, __nv_bfloat16* out,
                                                        int64_t np) {
  __shared__ uint16_t tile[64][64 + 2];
  const int64_t bh = blockIdx.z;
  const int64_t b = bh / in.H, h = bh % in.H;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * 64;
  const int d0 = blockIdx.y * 64;
  const uint16_t* src = static_cast<const uint16_t*>(in.data) + b * in.stride_b + h * in.stride_h;
  // load: 64 rows x 64 d (8 x 16-byte chunks per row)
  for (int idx = threadIdx.x; idx < 64 * 8; idx += 256) {
    const int r = idx / 8, cch = idx % 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n0 + r < in.N)
      v = *reinterpret_cast<const uint4*>(src + (n0 + r) * in.stride_n + d0 + cch * 8);
    const uint16_t* e = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
    for (int k = 0; k < 8; ++k) tile[r][cch * 8 + k] = e[k];
  }
  __syncthreads();
  // store: 64 d-rows x 64 n (8 x 16-byte chunks per row)
  uint16_t* dst = reinterpret_cast<uint16_t*>(out) + (bh * in.D + d0) * np;
  for (int idx = threadIdx.x; idx < 64 * 8; idx += 256) {
    const int dr = idx / 8, cch = idx % 8;
    const int64_t n = n0 + cch * 8;
    if (n >= np) continue;
    union {
      uint16_t h[8];
      uint4 v;
    } e;
#pragma unroll
    for (int k = 0; k < 8; ++k) e.h[k] = tile[cch * 8 + k][dr];
    *reinterpret_cast<uint4*>(dst + dr * np + n) = e.v;
  }
}

}  // namespace

int64_t transposed_row_len(int64_t n) { return (n + 7) / 8 * 8; }

size_t transposed_bytes(const lsx_tensor& t) {
  return static_cast<size_t>(t.B * t.H * t.D * transposed_row_len(t.N)) * 2;
}

int launch_transpose(const lsx_tensor& in, void* out, cudaStream_t s) {
  if (in.N == 0) return LSX_OK;
  if (in.B * in.H > 65535 || in.D % 64 != 0) return LSX_ERR_UNSUPPORTED;
  const int64_t np = transposed_row_len(in.N);
  dim3 grid(static_cast<unsigned>(ceil_div(np, 64)), static_cast<unsigned>(in.D / 64),
            static_cast<unsigned>(in.B * in.H));
  timing_begin(kKidTranspose, s);
  transpose_kernel<<<grid, 256, 0, s>>>(in, static_cast<__nv_bfloat16*>(out), np);
  timing_end(kKidTranspose, s);
  return cudaGetLastError() == cudaSuccess ? LSX_OK : LSX_ERR_LAUNCH;
}

}  // namespace lsx
