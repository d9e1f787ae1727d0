// Transpose of a bf16 matrix, used by the backward of the linear logprob to put
// the operands of dL/dy = G . W and dL/dW = G^T . y in the K-major layout the
// tensor-core GEMM reads (K contiguous): W [V, d] -> W^T [d, V], y [T, d] ->
// y^T [d, T].  64 x 64 tiles staged in shared memory (padded rows: no bank
// conflicts), 16-byte loads and stores where the tile is whole.
#include "tim_common.cuh"

namespace tim {

constexpr int kTrTile = 64;

// in: [rows, cols] with row stride ld_in; out: [cols, rows] with row stride ld_out.
__global__ void __launch_bounds__(256)
    transpose_bf16_kernel(const uint16_t* __restrict__ in, int64_t rows, int64_t cols,
                          int64_t ld_in, uint16_t* __restrict__ out, int64_t ld_out) {
  __shared__ uint16_t tile[kTrTile][kTrTile + 2];
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTrTile;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTrTile;
  const int tx = threadIdx.x & 7;   // 8 groups of 8 columns
  const int ty = threadIdx.x >> 3;  // 32 rows per pass
  for (int rr = ty; rr < kTrTile; rr += 32) {
    const int64_t r = r0 + rr;
    const int64_t c = c0 + tx * 8;
    if (r < rows && c + 8 <= cols && ((ld_in & 7) == 0)) {
      const uint4 v = *reinterpret_cast<const uint4*>(in + r * ld_in + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        tile[rr][tx * 8 + 2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
        tile[rr][tx * 8 + 2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        tile[rr][tx * 8 + i] = (r < rows && c + i < cols) ? in[r * ld_in + c + i] : 0;
    }
  }
  __syncthreads();
  for (int cc = ty; cc < kTrTile; cc += 32) {
    const int64_t orow = c0 + cc;   // output row = input column
    const int64_t ocol = r0 + tx * 8;
    if (orow >= cols) continue;
    if (ocol + 8 <= rows && ((ld_out & 7) == 0)) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = static_cast<uint32_t>(tile[tx * 8 + 2 * i][cc]) |
               (static_cast<uint32_t>(tile[tx * 8 + 2 * i + 1][cc]) << 16);
      *reinterpret_cast<uint4*>(out + orow * ld_out + ocol) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (ocol + i < rows) out[orow * ld_out + ocol + i] = tile[tx * 8 + i][cc];
    }
  }
}

cudaError_t launch_transpose_bf16(const void* in, int64_t rows, int64_t cols, int64_t ld_in,
                                  void* out, int64_t ld_out, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((cols + kTrTile - 1) / kTrTile),
                  static_cast<unsigned>((rows + kTrTile - 1) / kTrTile));
  transpose_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(in), rows, cols,
                                                  ld_in, static_cast<uint16_t*>(out), ld_out);
  return cudaGetLastError();
}

}  // namespace tim
