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

// Loads of a lane's chunks are issued kLoadBatch at a time (chunks c, c + 32,
// ... of one batch in flight together); the arithmetic that follows keeps the
// chunk order, so the results do not depend on the batching.
constexpr int kLoadBatch = 8;

// Sum of squares of one row in the fixed order above; every lane returns the same
// value.
__device__ __forceinline__ float row_sum_squares(const uint4* h, int nvec, int lane) {
  float ss = 0.f;
  for (int c0 = lane; c0 < nvec; c0 += 32 * kLoadBatch) {
    uint4 v[kLoadBatch];
#pragma unroll
    for (int i = 0; i < kLoadBatch; ++i)
      if (c0 + 32 * i < nvec) v[i] = __ldg(h + c0 + 32 * i);
#pragma unroll
    for (int i = 0; i < kLoadBatch; ++i) {
      if (c0 + 32 * i >= nvec) break;
      float f[8];
      unpack_bf16x8(v[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(f[j], f[j], ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  return ss;
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

  const float ss = row_sum_squares(h, nvec, lane);
  if (!isfinite(ss)) {
    if (lane == 0) set_status(status, TIM_ERR_NONFINITE);
  }
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);

  for (int c0 = lane; c0 < nvec; c0 += 32 * kLoadBatch) {
    uint4 hv[kLoadBatch], gv[kLoadBatch];
#pragma unroll
    for (int k = 0; k < kLoadBatch; ++k)
      if (c0 + 32 * k < nvec) {
        hv[k] = __ldg(h + c0 + 32 * k);
        gv[k] = __ldg(gamma + c0 + 32 * k);
      }
#pragma unroll
    for (int k = 0; k < kLoadBatch; ++k) {
      const int c = c0 + 32 * k;
      if (c >= nvec) break;
      float f[8], g[8];
      unpack_bf16x8(hv[k], f);
      unpack_bf16x8(gv[k], g);
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
}

// FP32 head: the same RMSNorm with y kept in fp32 (no bf16 rounding), written as
// a tf32 part (the low 13 mantissa bits cleared) and the remainder y - big,
// which fp32 holds exactly.  Rows T .. T_pad-1 are written as zeros.
__global__ void __launch_bounds__(32 * kNormRowsPerBlock)
    rmsnorm_rows_split_kernel(const uint4* __restrict__ hidden, const uint4* __restrict__ gamma,
                              int64_t T, int64_t T_pad, int d, float eps,
                              float4* __restrict__ ybig, float4* __restrict__ ysmall,
                              int* status) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNormRowsPerBlock + warp;
  if (row >= T_pad) return;
  const int nvec = d >> 3;
  float4* ob = ybig + row * (2 * nvec);
  float4* os = ysmall + row * (2 * nvec);
  if (row >= T) {
    for (int c = lane; c < 2 * nvec; c += 32) {
      ob[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      os[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const uint4* h = hidden + row * nvec;
  const float ss = row_sum_squares(h, nvec, lane);
  if (!isfinite(ss)) {
    if (lane == 0) set_status(status, TIM_ERR_NONFINITE);
  }
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  for (int c = lane; c < nvec; c += 32) {
    float f[8], g[8], b[8], r[8];
    unpack_bf16x8(__ldg(h + c), f);
    unpack_bf16x8(__ldg(gamma + c), g);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // __fmul_rn: the product must be rounded before the subtraction below
      // (no contraction into a fused multiply-add).
      const float y = __fmul_rn(__fmul_rn(f[i], rstd), g[i]);
      b[i] = __uint_as_float(__float_as_uint(y) & 0xFFFFE000u);
      r[i] = y - b[i];
    }
    ob[2 * c] = make_float4(b[0], b[1], b[2], b[3]);
    ob[2 * c + 1] = make_float4(b[4], b[5], b[6], b[7]);
    os[2 * c] = make_float4(r[0], r[1], r[2], r[3]);
    os[2 * c + 1] = make_float4(r[4], r[5], r[6], r[7]);
  }
}

// Elementwise tf32 split of fp32 values: big = x with the low 13 mantissa bits
// cleared, small = x - big (exact).  n4 = number of float4 groups.
__global__ void split_tf32_kernel(const float4* __restrict__ x, int64_t n4,
                                  float4* __restrict__ big, float4* __restrict__ small) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = __ldg(x + i);
    float4 b;
    b.x = __uint_as_float(__float_as_uint(v.x) & 0xFFFFE000u);
    b.y = __uint_as_float(__float_as_uint(v.y) & 0xFFFFE000u);
    b.z = __uint_as_float(__float_as_uint(v.z) & 0xFFFFE000u);
    b.w = __uint_as_float(__float_as_uint(v.w) & 0xFFFFE000u);
    big[i] = b;
    small[i] = make_float4(v.x - b.x, v.y - b.y, v.z - b.z, v.w - b.w);
  }
}

// ---------------------------------------------------------------------------
// RMSNorm backward (the bf16 rounding of y passed straight through).  With
// r = rstd (recomputed exactly as the forward computes it):
//   dh_ti    = r_t gamma_i dy_ti - (r_t^3 / d) h_ti s_t,  s_t = sum_j gamma_j dy_tj h_tj
//   dgamma_i = sum_t dy_ti h_ti r_t
// Rows: one warp per row, s_t in the forward's lane / butterfly order.  dgamma:
// per-column sums over chunks of kDgRows rows (rows in order), then the chunk
// partials folded in chunk order -- deterministic for a given batch.
constexpr int kDgRows = 256;

__global__ void __launch_bounds__(32 * kNormRowsPerBlock)
    rmsnorm_backward_rows_kernel(const uint4* __restrict__ hidden, const uint4* __restrict__ gamma,
                                 const float4* __restrict__ dy, int64_t T, int d, float eps,
                                 float4* __restrict__ dh, float* __restrict__ rstd_out,
                                 int* status) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNormRowsPerBlock + warp;
  if (row >= T) return;
  const int nvec = d >> 3;
  const uint4* h = hidden + row * nvec;
  const float4* g = dy + row * (2 * nvec);
  const float ss = row_sum_squares(h, nvec, lane);
  if (!isfinite(ss)) {
    if (lane == 0) set_status(status, TIM_ERR_NONFINITE);
  }
  const float rstd = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  float sgd = 0.f;
  for (int c = lane; c < nvec; c += 32) {
    float f[8], w[8];
    unpack_bf16x8(__ldg(h + c), f);
    unpack_bf16x8(__ldg(gamma + c), w);
    const float4 a = __ldg(g + 2 * c), b = __ldg(g + 2 * c + 1);
    const float gv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) sgd = fmaf(w[i] * gv[i], f[i], sgd);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sgd += __shfl_xor_sync(0xFFFFFFFFu, sgd, o);
  const float coef = rstd * rstd * rstd / static_cast<float>(d) * sgd;
  float4* out = dh + row * (2 * nvec);
  for (int c = lane; c < nvec; c += 32) {
    float f[8], w[8];
    unpack_bf16x8(__ldg(h + c), f);
    unpack_bf16x8(__ldg(gamma + c), w);
    const float4 a = __ldg(g + 2 * c), b = __ldg(g + 2 * c + 1);
    const float gv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = rstd * w[i] * gv[i] - coef * f[i];
    out[2 * c] = make_float4(o[0], o[1], o[2], o[3]);
    out[2 * c + 1] = make_float4(o[4], o[5], o[6], o[7]);
  }
  if (lane == 0) rstd_out[row] = rstd;
}

// partial[chunk][i] = sum over the chunk's rows (in order) of dy_ti h_ti r_t
__global__ void __launch_bounds__(256)
    dgamma_partial_kernel(const uint16_t* __restrict__ hidden, const float* __restrict__ dy,
                          const float* __restrict__ rstd, int64_t T, int d,
                          float* __restrict__ partial) {
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i >= d) return;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kDgRows;
  const int64_t t1 = t0 + kDgRows < T ? t0 + kDgRows : T;
  float acc = 0.f;
  for (int64_t t = t0; t < t1; ++t) {
    const float hv = __uint_as_float(static_cast<uint32_t>(__ldg(hidden + t * d + i)) << 16);
    acc = fmaf(__ldg(dy + t * d + i) * hv, __ldg(rstd + t), acc);
  }
  partial[static_cast<int64_t>(blockIdx.y) * d + i] = acc;
}

__global__ void __launch_bounds__(256)
    dgamma_fold_kernel(const float* __restrict__ partial, int n_chunks, int d, float* dgamma,
                       int accumulate) {
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i >= d) return;
  float acc = 0.f;
  for (int c = 0; c < n_chunks; ++c) acc += partial[static_cast<int64_t>(c) * d + i];
  dgamma[i] = accumulate ? dgamma[i] + acc : acc;
}

int rmsnorm_backward_chunks(int64_t T) { return static_cast<int>((T + kDgRows - 1) / kDgRows); }

cudaError_t launch_rmsnorm_backward(const void* hidden, const void* gamma, const float* dy,
                                    int64_t T, int d, float eps, float* dh, float* dgamma,
                                    int accumulate, float* rstd, float* partial, int* status,
                                    cudaStream_t stream) {
  const int64_t blocks = (T + kNormRowsPerBlock - 1) / kNormRowsPerBlock;
  rmsnorm_backward_rows_kernel<<<static_cast<unsigned>(blocks), 32 * kNormRowsPerBlock, 0,
                                 stream>>>(static_cast<const uint4*>(hidden),
                                           static_cast<const uint4*>(gamma),
                                           reinterpret_cast<const float4*>(dy), T, d, eps,
                                           reinterpret_cast<float4*>(dh), rstd, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nc = rmsnorm_backward_chunks(T);
  const dim3 grid(static_cast<unsigned>((d + 255) / 256), static_cast<unsigned>(nc));
  dgamma_partial_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(hidden), dy, rstd,
                                                  T, d, partial);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  dgamma_fold_kernel<<<static_cast<unsigned>((d + 255) / 256), 256, 0, stream>>>(partial, nc, d,
                                                                                 dgamma, accumulate);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_rows_split(const void* hidden, const void* gamma, int64_t T, int d,
                                      float eps, float* ybig, float* ysmall, int* status,
                                      cudaStream_t stream) {
  const int64_t T_pad = rows_padded(T);
  const int64_t blocks = (T_pad + kNormRowsPerBlock - 1) / kNormRowsPerBlock;
  rmsnorm_rows_split_kernel<<<static_cast<unsigned>(blocks), 32 * kNormRowsPerBlock, 0, stream>>>(
      static_cast<const uint4*>(hidden), static_cast<const uint4*>(gamma), T, T_pad, d, eps,
      reinterpret_cast<float4*>(ybig), reinterpret_cast<float4*>(ysmall), status);
  return cudaGetLastError();
}

cudaError_t launch_split_tf32(const float* x, int64_t n, float* big, float* small,
                              cudaStream_t stream, int num_sms) {
  const int64_t n4 = n / 4;
  int64_t blocks = (n4 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  split_tf32_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(x), n4, reinterpret_cast<float4*>(big),
      reinterpret_cast<float4*>(small));
  return cudaGetLastError();
}

// Loads rmsnorm_rows_kernel on the current device now (the runtime loads kernels
// lazily, and loading takes device memory).
cudaError_t load_rmsnorm_rows_kernel() {
  cudaFuncAttributes attr;
  return cudaFuncGetAttributes(&attr, rmsnorm_rows_kernel);
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
