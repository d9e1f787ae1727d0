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

// Fold records t0 .. t1-1 (t0 < t1) of one row left to right; records are
// fetched kFoldBatch at a time so the loads overlap (the merge order is
// unchanged).  A 151936-column vocabulary has 594 tiles, 38 per range: two
// batches, i.e. two round trips to memory per range.
constexpr int kFoldBatch = 20;

__device__ __forceinline__ Rec fold_range(const float4* p, int t0, int t1) {
  Rec acc = {0.f, 0.f, 0.f, 0};
  for (int t = t0; t < t1; t += kFoldBatch) {
    Rec buf[kFoldBatch];
#pragma unroll
    for (int i = 0; i < kFoldBatch; ++i)
      if (t + i < t1) buf[i] = load_rec(p + static_cast<int64_t>(t + i) * 32);
#pragma unroll
    for (int i = 0; i < kFoldBatch; ++i)
      if (t + i < t1) acc = (t + i == t0) ? buf[i] : merge(acc, buf[i]);
  }
  return acc;
}

__device__ __forceinline__ float lse_from(const Rec& r) {
  return (r.m + log2f(r.s)) * 0.69314718055994531f;
}

__global__ void __launch_bounds__(32 * kFinWarps)
    lse_finalize_kernel(const float4* __restrict__ part, const float* __restrict__ tgt,
                        const int32_t* __restrict__ ids, int64_t T, int V, int n_tiles,
                        float* __restrict__ out_lp, float* __restrict__ out_lse,
                        int32_t* __restrict__ out_top1, int* status) {
  __shared__ Rec red[kFinWarps][32];
  // launched with programmatic stream serialisation: the launch overlaps the
  // LM-head kernel's tail, and the records are read only after it has completed
  pdl_wait();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t group = blockIdx.x;
  const int per = (n_tiles + kFinWarps - 1) / kFinWarps;
  const int t0 = warp * per;
  const int t1 = min(n_tiles, t0 + per);
  const float4* p = part + group * static_cast<int64_t>(n_tiles) * 32 + lane;

  if (t0 < t1) red[warp][lane] = fold_range(p, t0, t1);
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
  const float lse = lse_from(r);
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

// Loads lse_finalize_kernel on the current device now (the runtime loads kernels
// lazily, and loading takes device memory).
cudaError_t load_lse_finalize_kernel() {
  cudaFuncAttributes attr;
  return cudaFuncGetAttributes(&attr, lse_finalize_kernel);
}

cudaError_t launch_lse_finalize(const void* part, const float* tgt, const int32_t* ids, int64_t T,
                                int V, float* out_lp, float* out_lse, int32_t* out_top1,
                                int* status, cudaStream_t stream) {
  const int n_tiles = (V + kBN - 1) / kBN;
  const int64_t groups = (T + kRowGroup - 1) / kRowGroup;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(groups));
  cfg.blockDim = dim3(32 * kFinWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_finalize_kernel, static_cast<const float4*>(part), tgt, ids,
                            T, V, n_tiles, out_lp, out_lse, out_top1, status);
}

// ---------------------------------------------------------------------------
// Vocabulary-parallel form of the same merge.
//
// "Debugging Logprob Mismatches ...", Collect A/B and C in Your Own Run: a
// vocabulary-parallel head must normalise over all shards together; "Training
// and rollout stop disagreeing ...", Interpretation: cross-rank LSE merge with
// a fixed rank reduction order.  The vocabulary is cut along the 16 fixed
// merge ranges above: with G ranks (G = 1, 2, 4, 8 or 16) rank g owns the
// L = 16 / G consecutive ranges g*L .. g*L+L-1 (whole 256-column tiles).
// Rank g folds its ranges and applies the tree levels with stride < L
// (lse_shard_reduce_kernel); after an all-gather of the per-row records, the
// levels with stride >= L run over the G records in rank order
// (lse_merge_shards_kernel).  Every merge is the one the unsharded kernel
// performs, in the same order, so the outputs are bitwise identical to the
// unsharded path's for every G.

__host__ __device__ inline int ranges_per(int n_tiles) {
  return (n_tiles + kFinWarps - 1) / kFinWarps;
}

__global__ void __launch_bounds__(32 * kFinWarps)
    lse_shard_reduce_kernel(const float4* __restrict__ part, const float* __restrict__ tgt,
                            int64_t T, int n_tiles, int n_tiles_shard, int g, int L,
                            float4* __restrict__ out_rec, float* __restrict__ out_tgt) {
  __shared__ Rec red[kFinWarps][32];
  const int warp = threadIdx.x >> 5;  // local range index, 0 .. L-1
  const int lane = threadIdx.x & 31;
  const int64_t group = blockIdx.x;
  const int per = ranges_per(n_tiles);
  const int w = g * L + warp;         // global range index
  const int base = g * L * per;       // global tile index of the shard's first tile
  const int t0 = w * per;
  const int t1 = min(n_tiles, t0 + per);
  const float4* p = part + group * static_cast<int64_t>(n_tiles_shard) * 32 + lane;
  if (t0 < t1) red[warp][lane] = fold_range(p, t0 - base, t1 - base);
  __syncthreads();
  for (int stride = 1; stride < L; stride <<= 1) {
    if ((warp & (2 * stride - 1)) == 0 && (w + stride) * per < n_tiles) {
      red[warp][lane] = merge(red[warp][lane], red[warp + stride][lane]);
    }
    __syncthreads();
  }
  if (warp != 0) return;
  const int64_t row = group * 32 + lane;
  if (row >= T) return;
  const Rec r = red[0][lane];
  out_rec[row] = make_float4(r.m, r.s, r.z, __int_as_float(r.id));
  out_tgt[row] = __ldg(tgt + row);
}

__global__ void __launch_bounds__(128)
    lse_merge_shards_kernel(const float4* __restrict__ recs, const float* __restrict__ tgts,
                            const int32_t* __restrict__ ids, int64_t T, int V, int G, int L,
                            int n_tiles, float* __restrict__ out_lp, float* __restrict__ out_lse,
                            int32_t* __restrict__ out_top1, int* status) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= T) return;
  const int per = ranges_per(n_tiles);
  Rec r[kFinWarps];
  for (int k = 0; k < G; ++k) r[k] = load_rec(recs + static_cast<int64_t>(k) * T + row);
  for (int stride = 1; stride < G; stride <<= 1) {
    for (int k = 0; k + stride < G; k += 2 * stride) {
      if ((k + stride) * L * per < n_tiles) r[k] = merge(r[k], r[k + stride]);
    }
  }
  const float lse = lse_from(r[0]);
  const int x = __ldg(ids + row);
  float lp;
  if (x >= 0 && x < V) {
    const int owner = (x / kBN) / per / L;
    lp = __ldg(tgts + static_cast<int64_t>(owner) * T + row) - lse;
  } else {
    lp = __int_as_float(0x7FC00000);
    set_status(status, TIM_ERR_TOKEN_RANGE);
  }
  if (!isfinite(lse)) set_status(status, TIM_ERR_NONFINITE);
  out_lp[row] = lp;
  out_lse[row] = lse;
  out_top1[row] = r[0].id;
}

// Shard g of G: global tiles [g*L*per, min(n_tiles, (g+1)*L*per)).
__host__ void vocab_shard_range(int V, int G, int g, int* v0, int* v_len) {
  const int n_tiles = (V + kBN - 1) / kBN;
  const int per = ranges_per(n_tiles);
  const int L = kFinWarps / G;
  const long long t0 = static_cast<long long>(g) * L * per;
  const long long t1 = static_cast<long long>(g + 1) * L * per;
  const long long c0 = t0 * kBN;
  const long long c1 = t1 * kBN < V ? t1 * kBN : V;
  *v0 = static_cast<int>(c0 < V ? c0 : V);
  *v_len = static_cast<int>(c1 > c0 ? c1 - c0 : 0);
}

cudaError_t launch_shard_reduce(const void* part, const float* tgt, int64_t T, int V, int G, int g,
                                int v_len, void* out_rec, float* out_tgt, cudaStream_t stream) {
  const int n_tiles = (V + kBN - 1) / kBN;
  const int n_tiles_shard = (v_len + kBN - 1) / kBN;
  const int L = kFinWarps / G;
  const int64_t groups = (T + kRowGroup - 1) / kRowGroup;
  lse_shard_reduce_kernel<<<static_cast<unsigned>(groups), 32 * L, 0, stream>>>(
      static_cast<const float4*>(part), tgt, T, n_tiles, n_tiles_shard, g, L,
      static_cast<float4*>(out_rec), out_tgt);
  return cudaGetLastError();
}

cudaError_t launch_merge_shards(const void* recs, const float* tgts, const int32_t* ids, int64_t T,
                                int V, int G, float* out_lp, float* out_lse, int32_t* out_top1,
                                int* status, cudaStream_t stream) {
  const int n_tiles = (V + kBN - 1) / kBN;
  const int L = kFinWarps / G;
  const int64_t blocks = (T + 127) / 128;
  lse_merge_shards_kernel<<<static_cast<unsigned>(blocks), 128, 0, stream>>>(
      static_cast<const float4*>(recs), tgts, ids, T, V, G, L, n_tiles, out_lp, out_lse,
      out_top1, status);
  return cudaGetLastError();
}

}  // namespace tim
