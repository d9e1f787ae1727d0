// Processed (top-k, then top-p) selected-token logprob.
//
// "Debugging Logprob Mismatches in LLM Reinforcement Learning", Make Sure Both
// Scores Describe the Same Probability: a sampler's score is taken on the
// distribution left after its filters, renormalised (top-k with k = 2 turns
// (0.50, 0.30, 0.20) into (0.625, 0.375, 0)).  Order: temperature, top-k (ties
// keep the lower token id), top-p on the renormalised top-k distribution
// (keep tokens whose preceding cumulative probability is < p).  A filtered-out
// target scores -inf.
//
// Steps:
//  1. the LM-head kernel in top-4 mode: for every (row, 256-column tile) the four
//     largest logits and their ids;
//  2. topk_candidates_kernel, one warp per row: thr = the k-th largest tile
//     maximum (bitwise radix select on order-preserving keys).  The k largest
//     tile maxima are k distinct logits, so every top-k logit is >= thr, and a
//     logit >= thr can only sit in a tile whose maximum is >= thr.  If in each
//     such tile the 4th largest logit is < thr, the stored top-4 lists hold every
//     logit >= thr: they become the row's candidates.  Otherwise (a tile with
//     four or more logits >= thr, or a vocabulary with fewer than k tiles) the
//     row goes on a fallback list;
//  3. the fallback rows are gathered and the LM-head kernel runs again over them
//     in candidate mode (every logit >= thr appended), scheduling only the row
//     tiles that hold them;
//  4. topk_finalize_kernel: per row, the candidates are sorted by (logit
//     descending, id ascending) with a warp bitonic sort; the first k form the
//     top-k set; the fp64 exponentials of the top-k are taken in parallel (one
//     or two per lane), then one lane walks them in order for top-p and the
//     score.
// Both routes produce the same candidate set (all logits >= thr, the same fp32
// values from the same MMA sequence), so a row's result does not depend on
// which route it took or on the batch.
#include <cmath>

#include "tim_common.cuh"

namespace tim {

constexpr int kProcWarps = 4;
constexpr int kProcSortMax = TIM_PROCESSED_CAPACITY;  // elements per warp sort

// Bitonic sort of n2 (power of two) 64-bit keys, descending, by one warp.
// Each phase visits its n2 / 2 compare-exchange pairs directly (pair idx -> lower
// index i: a zero bit inserted at the stride's bit).
__device__ __forceinline__ void warp_sort_desc_u64(unsigned long long* b, int n2, int lane) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int idx = lane; idx < (n2 >> 1); idx += 32) {
        const int i = ((idx & ~(j - 1)) << 1) | (idx & (j - 1));
        const int ixj = i + j;
        const unsigned long long x = b[i], y = b[ixj];
        const bool down = (i & k) == 0;
        if ((x < y) == down) {
          b[i] = y;
          b[ixj] = x;
        }
      }
      __syncwarp();
    }
  }
}

// Monotone map of float bits to unsigned (larger float -> larger key).
__device__ __forceinline__ uint32_t ordered_bits(uint32_t f) {
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

constexpr int kThrPerLane = (TIM_PROCESSED_CAPACITY + 31) / 32;  // tile maxima per lane

__global__ void __launch_bounds__(32 * kProcWarps)
    topk_candidates_kernel(const Top4Rec* __restrict__ top4, int64_t T, int n_tiles, int k,
                           float* __restrict__ thr, int* __restrict__ cnt,
                           uint2* __restrict__ cand, int cap, int* __restrict__ fb_count,
                           int* __restrict__ fb_rows) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kProcWarps + warp;
  if (row >= T) return;
  if (n_tiles < k) {  // every logit is a candidate: the collect pass takes the row
    if (lane == 0) {
      thr[row] = -INFINITY;
      cnt[row] = 0;
      fb_rows[atomicAdd(fb_count, 1)] = static_cast<int>(row);
    }
    return;
  }
  const Top4Rec* rec = top4 + (row >> 5) * static_cast<int64_t>(n_tiles) * 32 + (row & 31);
  const int nr = (n_tiles + 31) / 32;  // rounds of 32 tiles actually present
  uint32_t key[kThrPerLane];
#pragma unroll
  for (int r = 0; r < kThrPerLane; ++r) {
    const int i = lane + 32 * r;
    key[r] = (r < nr && i < n_tiles)
                 ? ordered_bits(__float_as_uint(__ldg(&rec[static_cast<int64_t>(i) * 32].v[0])))
                 : 0u;
  }
  // the k-th largest tile maximum, one bit at a time from the top
  uint32_t prefix = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t candk = prefix | (1u << b);
    int c = 0;
#pragma unroll
    for (int r = 0; r < kThrPerLane; ++r)
      if (r < nr) c += key[r] >= candk ? 1 : 0;
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    if (c >= k) prefix = candk;
  }
  const float t = __uint_as_float((prefix & 0x80000000u) ? (prefix & 0x7FFFFFFFu) : ~prefix);
  // count this lane's candidates; a tile with four logits >= t may hold more
  int mine = 0, ovf = 0;
#pragma unroll
  for (int r = 0; r < kThrPerLane; ++r) {
    const int i = lane + 32 * r;
    if (r < nr && i < n_tiles) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(rec[static_cast<int64_t>(i) * 32].v));
      if (v.x >= t) {
        mine += 1 + (v.y >= t ? 1 : 0) + (v.z >= t ? 1 : 0) + (v.w >= t ? 1 : 0);
        ovf |= v.w >= t ? 1 : 0;
      }
    }
  }
  const int total = __reduce_add_sync(0xFFFFFFFFu, mine);
  if (__any_sync(0xFFFFFFFFu, ovf) || total > cap) {
    if (lane == 0) {
      thr[row] = t;
      cnt[row] = 0;
      fb_rows[atomicAdd(fb_count, 1)] = static_cast<int>(row);
    }
    return;
  }
  int off = mine;  // exclusive prefix over lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, off, o);
    if (lane >= o) off += u;
  }
  off -= mine;
  uint2* dst = cand + row * cap;
#pragma unroll
  for (int r = 0; r < kThrPerLane; ++r) {
    const int i = lane + 32 * r;
    if (r < nr && i < n_tiles) {
      const Top4Rec& q = rec[static_cast<int64_t>(i) * 32];
      const float4 v = __ldg(reinterpret_cast<const float4*>(q.v));
      if (v.x >= t) {
        const int4 id = __ldg(reinterpret_cast<const int4*>(q.id));
        dst[off++] = make_uint2(__float_as_uint(v.x), static_cast<uint32_t>(id.x));
        if (v.y >= t) dst[off++] = make_uint2(__float_as_uint(v.y), static_cast<uint32_t>(id.y));
        if (v.z >= t) dst[off++] = make_uint2(__float_as_uint(v.z), static_cast<uint32_t>(id.z));
      }
    }
  }
  if (lane == 0) {
    thr[row] = t;
    cnt[row] = total;
  }
}

// Copies the fallback rows of y (bf16 [*, d]) into consecutive rows of y_fb.
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint4* __restrict__ y, const int* __restrict__ fb_rows,
                       const int* __restrict__ fb_count, int nvec, uint4* __restrict__ y_fb) {
  const int n = __ldcg(fb_count);
  for (int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < n;
       w += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    const int64_t src = __ldcg(fb_rows + w);
    for (int c = threadIdx.x & 31; c < nvec; c += 32) y_fb[w * nvec + c] = __ldg(y + src * nvec + c);
  }
}

__global__ void __launch_bounds__(32 * kProcWarps)
    topk_finalize_kernel(const uint2* __restrict__ cand, const int* __restrict__ cnt,
                         const int32_t* __restrict__ ids, int64_t T, int V, int k, double top_p,
                         double temperature, int cap, float* __restrict__ out_lp,
                         float* __restrict__ out_lse, int32_t* __restrict__ out_kept,
                         int32_t* __restrict__ head_ids, float* __restrict__ head_lp,
                         int* status) {
  extern __shared__ unsigned long long sbuf[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kProcWarps + warp;
  if (row >= T) return;
  const int n = __ldcg(cnt + row);
  const int x = __ldg(ids + row);
  const int kh = k < V ? k : V;  // head entries per row
  if (n > cap || n < 1) {
    if (lane == 0) {
      set_status(status, n > cap ? TIM_ERR_CAPACITY : TIM_ERR_NONFINITE);
      out_lp[row] = __int_as_float(0x7FC00000);
      out_lse[row] = __int_as_float(0x7FC00000);
      out_kept[row] = 0;
    }
    if (head_ids != nullptr)
      for (int i = lane; i < kh; i += 32) {
        head_ids[row * kh + i] = -1;
        head_lp[row * kh + i] = __int_as_float(0x7FC00000);
      }
    return;
  }
  unsigned long long* b = sbuf + warp * kProcSortMax;
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  const uint2* c = cand + row * cap;
  for (int i = lane; i < n2; i += 32) {
    if (i < n) {
      const uint2 v = __ldcg(c + i);
      b[i] = (static_cast<unsigned long long>(ordered_bits(v.x)) << 32) |
             static_cast<unsigned long long>(0xFFFFFFFFu - v.y);
    } else {
      b[i] = 0ull;
    }
  }
  __syncwarp();
  warp_sort_desc_u64(b, n2, lane);
  __syncwarp();

  const int kk = k < n ? k : n;
  // scaled logits and exp(s_i - s_0) of the top-k, two entries per lane at most
  // (k <= 64), written back over the sorted keys as doubles
  double* ev = reinterpret_cast<double*>(b);
  int* idv_s = reinterpret_cast<int*>(b + TIM_PROCESSED_MAX_K * 2);
  const uint32_t key0 = static_cast<uint32_t>(b[0] >> 32);
  const double m =
      static_cast<double>(__uint_as_float((key0 & 0x80000000u) ? (key0 & 0x7FFFFFFFu) : ~key0)) /
      temperature;
  double sv[2], evv[2];
  int idl[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    if (i < kk) {
      const uint32_t key = static_cast<uint32_t>(b[i] >> 32);
      const uint32_t fb = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
      sv[h] = static_cast<double>(__uint_as_float(fb)) / temperature;
      idl[h] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(b[i] & 0xFFFFFFFFull));
      evv[h] = exp(sv[h] - m);
    }
  }
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    if (i < kk) {
      ev[i] = evv[h];
      ev[TIM_PROCESSED_MAX_K + i] = sv[h];
      idv_s[i] = idl[h];
    }
  }
  __syncwarp();
  if (lane != 0) return;
  const double* s = ev + TIM_PROCESSED_MAX_K;  // scaled logits of the top-k, in order
  const int* idv = idv_s;                      // their token ids
  double total = 0.0;
  for (int i = 0; i < kk; ++i) total += ev[i];
  // top-p on the renormalised top-k distribution
  int kept = 0;
  double before = 0.0, kept_sum = 0.0;
  for (int i = 0; i < kk; ++i) {
    const double e = ev[i];
    if (i > 0 && !(before < top_p * total)) break;
    kept_sum += e;
    before += e;
    ++kept;
  }
  const double lse = m + log(kept_sum);
  double lp = -INFINITY;
  if (x < 0 || x >= V) {
    lp = NAN;
    set_status(status, TIM_ERR_TOKEN_RANGE);
  } else {
    for (int i = 0; i < kept; ++i)
      if (idv[i] == x) lp = s[i] - lse;
  }
  if (!isfinite(lse)) set_status(status, TIM_ERR_NONFINITE);
  out_lp[row] = static_cast<float>(lp);
  out_lse[row] = static_cast<float>(lse);
  out_kept[row] = kept;
  if (head_ids != nullptr) {
    // the top-k head: ids in top-k order, processed logprobs (-inf past the top-p cut)
    for (int i = 0; i < kh; ++i) {
      head_ids[row * kh + i] = i < kk ? idv[i] : -1;
      head_lp[row * kh + i] = i < kept ? static_cast<float>(s[i] - lse) : -INFINITY;
    }
  }
}

cudaError_t launch_topk_candidates(const void* top4, int64_t T, int V, int k, float* thr,
                                   int* cnt, void* cand, int cap, int* fb_count, int* fb_rows,
                                   cudaStream_t stream) {
  const int n_tiles = (V + kBN - 1) / kBN;
  const int64_t blocks = (T + kProcWarps - 1) / kProcWarps;
  topk_candidates_kernel<<<static_cast<unsigned>(blocks), 32 * kProcWarps, 0, stream>>>(
      static_cast<const Top4Rec*>(top4), T, n_tiles, k, thr, cnt, static_cast<uint2*>(cand), cap,
      fb_count, fb_rows);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* y, const int* fb_rows, const int* fb_count, int64_t T,
                               int d, void* y_fb, cudaStream_t stream, int num_sms) {
  int64_t blocks = (T * 32 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint4*>(y), fb_rows, fb_count, d / 8, static_cast<uint4*>(y_fb));
  return cudaGetLastError();
}

cudaError_t launch_topk_finalize(const void* cand, const int* cnt, const int32_t* ids, int64_t T,
                                 int V, int k, float top_p, float temperature, int cap,
                                 float* out_lp, float* out_lse, int32_t* out_kept,
                                 int32_t* head_ids, float* head_lp, int* status,
                                 cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kProcWarps) * kProcSortMax * 8;
  cudaError_t e = cudaFuncSetAttribute(topk_finalize_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t blocks = (T + kProcWarps - 1) / kProcWarps;
  topk_finalize_kernel<<<static_cast<unsigned>(blocks), 32 * kProcWarps, smem, stream>>>(
      static_cast<const uint2*>(cand), cnt, ids, T, V, k, static_cast<double>(top_p),
      static_cast<double>(temperature), cap, out_lp, out_lse, out_kept, head_ids, head_lp, status);
  return cudaGetLastError();
}

}  // namespace tim
