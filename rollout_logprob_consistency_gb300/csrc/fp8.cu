// FP8 (e4m3) quantisation of rows, one warp per row.
//
// "Rollout-Training Mismatch in LLM RL", section 3 (Unified FP8 table): FP8
// quantize-dequantize values and native FP8 GEMMs consuming codes and scales.
// Scaling: one power-of-two scale per row, the smallest s with
// max|row| / s <= 448 (1 for an all-zero row); codes = e4m3(x / s), rounded to
// nearest-even with saturation (CUDA's __nv_cvt_float_to_fp8).  A power-of-two
// scale makes x / s and the dequantisation s * code exact, so the GEMM on the
// codes with both scales applied after accumulation gives the logits of the
// quantize-dequantize operands.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "tim_common.cuh"

namespace tim {

constexpr int kQuantRowsPerBlock = 8;

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Exact power-of-two scale: amax = f 2^e (0.5 <= f < 1) and 448 = 0.875 2^9.
__device__ __forceinline__ int scale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int e = 0;
  const float f = frexpf(amax, &e);
  return f <= 0.875f ? e - 9 : e - 8;
}

__global__ void __launch_bounds__(32 * kQuantRowsPerBlock)
    quantize_rows_e4m3_kernel(const uint4* __restrict__ x, int64_t rows, int K,
                              uint2* __restrict__ codes, float* __restrict__ scales) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kQuantRowsPerBlock + warp;
  if (row >= rows) return;
  const int nvec = K >> 3;
  const uint4* xr = x + row * nvec;
  float amax = 0.f;
  for (int c = lane; c < nvec; c += 32) {
    float f[8];
    unpack8(__ldg(xr + c), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const int k = scale_exponent(amax);
  const float inv = ldexpf(1.f, -k);
  uint2* out = codes + row * nvec;
  for (int c = lane; c < nvec; c += 32) {
    float f[8];
    unpack8(__ldg(xr + c), f);
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b = __nv_cvt_float_to_fp8(f[i] * inv, __NV_SATFINITE, __NV_E4M3);
      w[i >> 2] |= (b & 0xFFu) << (8 * (i & 3));
    }
    out[c] = make_uint2(w[0], w[1]);
  }
  if (lane == 0) scales[row] = ldexpf(1.f, k);
}

cudaError_t launch_quantize_rows_e4m3(const void* x, int64_t rows, int K, void* codes,
                                      float* scales, cudaStream_t stream) {
  const int64_t blocks = (rows + kQuantRowsPerBlock - 1) / kQuantRowsPerBlock;
  quantize_rows_e4m3_kernel<<<static_cast<unsigned>(blocks), 32 * kQuantRowsPerBlock, 0,
                              stream>>>(static_cast<const uint4*>(x), rows, K,
                                        static_cast<uint2*>(codes), scales);
  return cudaGetLastError();
}

}  // namespace tim
