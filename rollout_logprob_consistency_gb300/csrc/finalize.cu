// Stage 3 of the linear logprob: merge each row's per-vocabulary-tile records
// into the full-vocabulary normaliser, in a fixed order.
//
// "Debugging Logprob Mismatches in LLM Reinforcement Learning", Collect A/B
// and C in Your Own Run: with a vocabulary-parallel head the normaliser must be
// taken over all shards together (normalising each shard alone scores a
// different distribution).  "Training and rollout stop disagreeing ...",
// Interpretation: the linear logprob covers the true vocabulary range and a
// cross-rank LSE merge.  Here the "shards" are the 256-column vocabulary tiles
// of the LM-head kernel, and the merge order is fixed:
//
//   the n_tiles records of a row are cut into 16 contiguous ranges (a function
//   of n_tiles only); warp w folds range w left to right; the 16 results are
//   combined by a balanced binary tree over w (strides 1, 2, 4, 8).
//
// Merge of two records covering lower (a) and higher (b) vocabulary ids, in
// the base-2 domain t = z * log2(e) / tau:
//   M = max(a.m, b.m),  s = a.s * 2^(a.m - M) + b.s * 2^(b.m - M),
//   best = b if b.z > a.z else a        (ties keep the lower id).
// Then lse = (M + log2 s) * ln 2 (nats) and logprob = s_x - lse, where s_x is
// the target's scaled logit written by the LM-head kernel.
#include "tim_common.cuh"

namespace tim {

constexpr int kFinWarps = 16;

struct Rec {
  float m, s, z;
  int id;
};

__device__ __forceinline__ Rec load_rec(const float4* p) {
  const float4 v = __ldg(p);
  return Rec{v.x, v.y, v.z, __float_as_int(v.w)};
}

__device__ __forceinline__ Rec merge(const Rec& a, const Rec& b) {
  Rec r;
  r.m = fmaxf(a.m, b.m);
  r.s = a.s * exp2f(a.m - r.m) + b.s * exp2f(b.m - r.m);
  if (b.z > a.z) {
    r.z = b.z;
    r.id = b.id;
  } else {
    r.z = a.z;
    r.id = a.id;
  }
  return r;
}

__global__ void __launch_bounds__(32 * kFinWarps)
    lse_finalize_kernel(const float4* __restrict__ part, const float* __restrict__ tgt,
                        const int32_t* __restrict__ ids, int64_t T, int V, int n_tiles,
                        float* __restrict__ out_lp, float* __restrict__ out_lse,
                        int32_t* __restrict__ out_top1, int* status) {
  __shared__ Rec red[kFinWarps][32];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t group = blockIdx.x;
  const int per = (n_tiles + kFinWarps - 1) / kFinWarps;
  const int t0 = warp * per;
  const int t1 = min(n_tiles, t0 + per);
  const float4* p = part + group * static_cast<int64_t>(n_tiles) * 32 + lane;

  if (t0 < t1) {
    // fold the range left to right; records are fetched 8 at a time so the
    // loads overlap (the merge order is unchanged)
    Rec acc = load_rec(p + static_cast<int64_t>(t0) * 32);
    for (int t = t0 + 1; t < t1; t += 8) {
      Rec buf[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (t + i < t1) buf[i] = load_rec(p + static_cast<int64_t>(t + i) * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (t + i < t1) acc = merge(acc, buf[i]);
    }
    red[warp][lane] = acc;
  }
  __syncthreads();
#pragma unroll
  for (int stride = 1; stride < kFinWarps; stride <<= 1) {
    if ((warp & (2 * stride - 1)) == 0 && (warp + stride) * per < n_tiles) {
      red[warp][lane] = merge(red[warp][lane], red[warp + stride][lane]);
    }
    __syncthreads();
  }
  if (warp != 0) return;
  const int64_t row = group * 32 + lane;
  if (row >= T) return;
  const Rec r = red[0][lane];
  const float lse = (r.m + log2f(r.s)) * 0.69314718055994531f;
  const int x = __ldg(ids + row);
  float lp;
  if (x >= 0 && x < V) {
    lp = __ldg(tgt + row) - lse;
  } else {
    lp = __int_as_float(0x7FC00000);  // quiet NaN
    set_status(status, TIM_ERR_TOKEN_RANGE);
  }
  if (!isfinite(lse)) set_status(status, TIM_ERR_NONFINITE);
  out_lp[row] = lp;
  out_lse[row] = lse;
  out_top1[row] = r.id;
}

cudaError_t launch_lse_finalize(const void* part, const float* tgt, const int32_t* ids, int64_t T,
                                int V, float* out_lp, float* out_lse, int32_t* out_top1,
                                int* status, cudaStream_t stream) {
  const int n_tiles = (V + kBN - 1) / kBN;
  const int64_t groups = (T + kRowGroup - 1) / kRowGroup;
  lse_finalize_kernel<<<static_cast<unsigned>(groups), 32 * kFinWarps, 0, stream>>>(
      static_cast<const float4*>(part), tgt, ids, T, V, n_tiles, out_lp, out_lse, out_top1,
      status);
  return cudaGetLastError();
}

}  // namespace tim
