// Stage 1 of the linear logprob: the final RMSNorm, one warp per row.
//
// "Training and rollout stop disagreeing: vime and RL-Kernel ...",
// Interpretation: the strict path pins the RMSNorm reduction domain and
// epsilon.  Here the domain is the full hidden size d, eps sits inside the
// square root, and the reduction order is fixed for every row:
//   lane l accumulates h^2 over its 8-element chunks l, l+32, l+64, ... in
//   order (fused multiply-add in fp32), then an xor butterfly over the 32 lanes
//   (offsets 16, 8, 4, 2, 1).
// Every lane ends with the same bits (IEEE addition is commutative), and the
// result depends only on the row's own values: the kernel is batch-invariant.
// y = bf16_rn((h * rstd) * gamma) in fp32, written for the LM-head GEMM; rows
// from T up to the next multiple of 128 are written as zeros (the GEMM reads
// whole 128-row tiles).
#include <cuda_bf16.h>

#include "tim_common.cuh"

namespace tim {

constexpr int kNormRowsPerBlock = 8;

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(32 * kNormRowsPerBlock)
    rmsnorm_rows_kernel(const uint4* __restrict__ hidden, const uint4* __restrict__ gamma,
                        int64_t T, int64_t T_pad, int d, float eps, uint4* __restrict__ y,
                        int* status) {
  pdl_launch_dependents();  // the LM-head kernel may start streaming W now
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNormRowsPerBlock + warp;
  if (row >= T_pad) return;
  const int nvec = d >> 3;
  uint4* out = y + row * nvec;
  if (row >= T) {
    for (int c = lane; c < nvec; c += 32) out[c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const uint4* h = hidden + row * nvec;

  float ss = 0.f;
  for (int c = lane; c < nvec; c += 32) {
    float f[8];
    unpack_bf16x8(__ldg(h + c), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);

  if (!isfinite(ss)) {
    if (lane == 0) set_status(status, TIM_ERR_NONFINITE);
  }
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);

  for (int c = lane; c < nvec; c += 32) {
    float f[8], g[8];
    unpack_bf16x8(__ldg(h + c), f);
    unpack_bf16x8(__ldg(gamma + c), g);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat16 lo = __float2bfloat16_rn((f[2 * i] * rstd) * g[2 * i]);
      const __nv_bfloat16 hi = __float2bfloat16_rn((f[2 * i + 1] * rstd) * g[2 * i + 1]);
      w[i] = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
    }
    out[c] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_rmsnorm_rows(const void* hidden, const void* gamma, int64_t T, int d,
                                float eps, void* y, int* status, cudaStream_t stream) {
  const int64_t T_pad = rows_padded(T);
  const int64_t blocks = (T_pad + kNormRowsPerBlock - 1) / kNormRowsPerBlock;
  rmsnorm_rows_kernel<<<static_cast<unsigned>(blocks), 32 * kNormRowsPerBlock, 0, stream>>>(
      static_cast<const uint4*>(hidden), static_cast<const uint4*>(gamma), T, T_pad, d, eps,
      static_cast<uint4*>(y), status);
  return cudaGetLastError();
}

}  // namespace tim
