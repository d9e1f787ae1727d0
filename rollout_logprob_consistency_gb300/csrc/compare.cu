// Three-way score comparison, one CTA per sequence (segmented reduction).
//
// Definitions (left minus right for the pairs A-B, B-C, A-C; A = generation,
// B = rollout replay, C = trainer forward):
//  - bitwise mismatch of float32 scores via their integer views, first
//    mismatching position and longest run, over active tokens only:
//    "Fault localization and mismatch bisect", Compare per-token logprobs and
//    Per-sequence observation patterns;
//  - signed mean, MAE and maximum absolute difference:
//    "Debugging Logprob Mismatches in LLM Reinforcement Learning", Check
//    Whether the Pattern Extends Across the Response, and the Metric
//    measurement basis (logprob_mae) of the Fault localization page;
//  - d = C - A, the exact split mean(C - A) = mean(C - B) + mean(B - A):
//    eq. (1) of "Rollout-Training Mismatch in LLM RL", section 1.2;
//  - Schulman k3 = exp(d) - 1 - d (evaluated as expm1(d) - d; overflow flagged,
//    never clipped): Metric measurement basis;
//  - token TIS weight min(exp(d), cap), zero on padding: "Rollout-Training
//    Mismatch in LLM RL", section 2.1, and "Diagnosing Training Inference
//    Mismatch in LLM Reinforcement Learning", 3. TIS.
//
// Each thread owns a 4-token vector (a 128-bit load of each score array when
// the arrays are 16-byte aligned) and walks its tokens in order.  Runs of
// differing tokens are combined with an ordered monoid
//   (n, ndiff, first, prefix_run, suffix_run, best_run)
// by a warp shuffle tree (lane i with lane i+o, o = 1, 2, 4, 8, 16) and then
// across the 8 warps in warp order, 1024 tokens at a time; counts, first
// position, runs and maxima are therefore exact, and the fp64 sums are taken in
// a fixed order.
#include <cmath>

#include "tim_common.cuh"

namespace tim {

constexpr int kCmpThreads = 256;
constexpr int kCmpWarps = kCmpThreads / 32;

template <typename I>
struct Runs {
  I n, ndiff, first, pre, suf, best;
};

template <typename I>
__device__ __forceinline__ Runs<I> runs_identity() {
  return Runs<I>{0, 0, -1, 0, 0, 0};
}

template <typename I, typename J>
__device__ __forceinline__ Runs<I> runs_combine(const Runs<I>& L, const Runs<J>& R) {
  Runs<I> o;
  o.n = L.n + R.n;
  o.ndiff = L.ndiff + R.ndiff;
  o.first = L.first >= 0 ? L.first : (R.first >= 0 ? L.n + R.first : static_cast<I>(-1));
  o.pre = (L.pre == L.n) ? L.n + R.pre : L.pre;
  o.suf = (R.suf == R.n) ? static_cast<I>(R.n) + L.suf : static_cast<I>(R.suf);
  I best = L.best > static_cast<I>(R.best) ? L.best : static_cast<I>(R.best);
  const I bridge = L.suf + static_cast<I>(R.pre);
  o.best = best > bridge ? best : bridge;
  return o;
}

__device__ __forceinline__ void runs_push(Runs<int>& r, bool diff) {
  const Runs<int> s{1, diff ? 1 : 0, diff ? 0 : -1, diff ? 1 : 0, diff ? 1 : 0, diff ? 1 : 0};
  r = runs_combine(r, s);
}

__device__ __forceinline__ Runs<int> warp_runs_reduce(Runs<int> r, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    Runs<int> x;
    x.n = __shfl_down_sync(0xFFFFFFFFu, r.n, o);
    x.ndiff = __shfl_down_sync(0xFFFFFFFFu, r.ndiff, o);
    x.first = __shfl_down_sync(0xFFFFFFFFu, r.first, o);
    x.pre = __shfl_down_sync(0xFFFFFFFFu, r.pre, o);
    x.suf = __shfl_down_sync(0xFFFFFFFFu, r.suf, o);
    x.best = __shfl_down_sync(0xFFFFFFFFu, r.best, o);
    if ((lane & (2 * o - 1)) == 0) r = runs_combine(r, x);
  }
  return r;
}

// Per-thread fp64 accumulators (fixed order within a thread).
struct Acc {
  double sgn[3], abs_[3], mx[3];
  double k3, tis;
  long long clipped;
  int flags;
};

__device__ __forceinline__ void token(Acc& acc, Runs<int> (&runs)[3], float a, float b, float c,
                                      double cap, double ln_cap, float* tis_w, int64_t t) {
  const uint32_t ia = __float_as_uint(a), ib = __float_as_uint(b), ic = __float_as_uint(c);
  if (!(isfinite(a) && isfinite(b) && isfinite(c))) acc.flags |= TIM_SEQ_NONFINITE;
  runs_push(runs[0], ia != ib);
  runs_push(runs[1], ib != ic);
  runs_push(runs[2], ia != ic);
  const double da = a, db = b, dc = c;
  const double x[3] = {da - db, db - dc, da - dc};
#pragma unroll
  for (int p = 0; p < 3; ++p) {
    acc.sgn[p] += x[p];
    acc.abs_[p] += fabs(x[p]);
    acc.mx[p] = fmax(acc.mx[p], fabs(x[p]));
  }
  const double d = dc - da;
  acc.k3 += expm1(d) - d;
  double w;
  if (d > ln_cap) {
    w = cap;
    acc.clipped += 1;
  } else {
    w = exp(d);
  }
  acc.tis += w;
  if (tis_w != nullptr) tis_w[t] = static_cast<float>(w);
}

template <bool kVec>
__global__ void __launch_bounds__(kCmpThreads)
    seg_compare_kernel(const float* __restrict__ A, const float* __restrict__ B,
                       const float* __restrict__ C, const int64_t* __restrict__ offs,
                       const uint8_t* __restrict__ mask, int64_t T, double cap, double ln_cap,
                       tim_seq_stats* __restrict__ out, float* __restrict__ tis_w, int* status) {
  __shared__ Runs<int> s_runs[kCmpWarps][3];
  __shared__ double s_red[kCmpWarps][11];
  __shared__ long long s_clip[kCmpWarps];
  __shared__ int s_flags[kCmpWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.x;
  const int64_t s = offs[j], e = offs[j + 1];
  tim_seq_stats st;
  if (!(s >= 0 && s <= e && e <= T)) {
    if (tid == 0) {
      memset(&st, 0, sizeof(st));
      for (int p = 0; p < 3; ++p) st.pair[p].first_div = -1;
      st.flags = TIM_SEQ_BAD_OFFSETS;
      out[j] = st;
      set_status(status, TIM_ERR_INVALID_ARG);
    }
    return;
  }

  Acc acc;
#pragma unroll
  for (int p = 0; p < 3; ++p) acc.sgn[p] = acc.abs_[p] = acc.mx[p] = 0.0;
  acc.k3 = acc.tis = 0.0;
  acc.clipped = 0;
  acc.flags = 0;
  Runs<long long> total[3] = {runs_identity<long long>(), runs_identity<long long>(),
                              runs_identity<long long>()};

  const int64_t vbeg = s >> 2, vend = (e + 3) >> 2;
  for (int64_t base = vbeg; base < vend; base += kCmpThreads) {
    Runs<int> runs[3] = {runs_identity<int>(), runs_identity<int>(), runs_identity<int>()};
    const int64_t v = base + tid;
    if (v < vend) {
      const int64_t t0 = v * 4;
      float av[4], bv[4], cv[4];
      uint8_t mv[4];
      if (kVec && t0 + 4 <= T) {
        const float4 a4 = __ldg(reinterpret_cast<const float4*>(A) + v);
        const float4 b4 = __ldg(reinterpret_cast<const float4*>(B) + v);
        const float4 c4 = __ldg(reinterpret_cast<const float4*>(C) + v);
        const uint32_t m4 = __ldg(reinterpret_cast<const uint32_t*>(mask) + v);
        av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
        bv[0] = b4.x; bv[1] = b4.y; bv[2] = b4.z; bv[3] = b4.w;
        cv[0] = c4.x; cv[1] = c4.y; cv[2] = c4.z; cv[3] = c4.w;
#pragma unroll
        for (int k = 0; k < 4; ++k) mv[k] = static_cast<uint8_t>((m4 >> (8 * k)) & 0xFFu);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int64_t t = t0 + k;
          const bool in = (t >= s && t < e);
          av[k] = in ? __ldg(A + t) : 0.f;
          bv[k] = in ? __ldg(B + t) : 0.f;
          cv[k] = in ? __ldg(C + t) : 0.f;
          mv[k] = in ? __ldg(mask + t) : 0;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t t = t0 + k;
        if (t < s || t >= e) continue;
        if (mv[k] > 1) acc.flags |= TIM_SEQ_BAD_MASK;
        if (mv[k] != 1) {
          if (tis_w != nullptr) tis_w[t] = 0.f;
          continue;
        }
        token(acc, runs, av[k], bv[k], cv[k], cap, ln_cap, tis_w, t);
      }
    }
#pragma unroll
    for (int p = 0; p < 3; ++p) {
      runs[p] = warp_runs_reduce(runs[p], lane);
      if (lane == 0) s_runs[warp][p] = runs[p];
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int p = 0; p < 3; ++p) {
        Runs<int> chunk = runs_identity<int>();
        for (int w = 0; w < kCmpWarps; ++w) chunk = runs_combine(chunk, s_runs[w][p]);
        total[p] = runs_combine(total[p], chunk);
      }
    }
    __syncthreads();
  }

  // fixed-order block reduction of the fp64 sums
  double v[11] = {acc.sgn[0], acc.sgn[1], acc.sgn[2], acc.abs_[0], acc.abs_[1], acc.abs_[2],
                  acc.mx[0],  acc.mx[1],  acc.mx[2],  acc.k3,      acc.tis};
  long long clip = acc.clipped;
  int flags = acc.flags;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int i = 0; i < 11; ++i) {
      const double other = __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
      v[i] = (i >= 6 && i < 9) ? fmax(v[i], other) : v[i] + other;
    }
    clip += __shfl_xor_sync(0xFFFFFFFFu, clip, o);
    flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, o);
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 11; ++i) s_red[warp][i] = v[i];
    s_clip[warp] = clip;
    s_flags[warp] = flags;
  }
  __syncthreads();
  if (tid != 0) return;
  for (int i = 0; i < 11; ++i) {
    double r = s_red[0][i];
    for (int w = 1; w < kCmpWarps; ++w)
      r = (i >= 6 && i < 9) ? fmax(r, s_red[w][i]) : r + s_red[w][i];
    v[i] = r;
  }
  clip = 0;
  flags = 0;
  for (int w = 0; w < kCmpWarps; ++w) {
    clip += s_clip[w];
    flags |= s_flags[w];
  }

  memset(&st, 0, sizeof(st));
  for (int p = 0; p < 3; ++p) st.pair[p].first_div = -1;
  const long long n = total[0].n;
  if (flags & TIM_SEQ_BAD_MASK) {
    st.flags = TIM_SEQ_BAD_MASK;
    set_status(status, TIM_ERR_BAD_MASK);
  } else if (n == 0) {
    st.flags = TIM_SEQ_EMPTY;
    set_status(status, TIM_ERR_EMPTY_SEQUENCE);
  } else {
    const double dn = static_cast<double>(n);
    st.n_valid = n;
    for (int p = 0; p < 3; ++p) {
      st.pair[p].mismatch_count = total[p].ndiff;
      st.pair[p].first_div = total[p].first;
      st.pair[p].longest_run = total[p].best;
      st.pair[p].max_abs_diff = v[6 + p];
      st.pair[p].signed_mean = v[p] / dn;
      st.pair[p].mae = v[3 + p] / dn;
    }
    st.mean_log_ratio = -v[2] / dn;
    st.mean_weight_move = -v[1] / dn;
    st.mean_same_version = -v[0] / dn;
    st.k3_mean = v[9] / dn;
    st.tis_mean = v[10] / dn;
    st.tis_clipped = clip;
    st.flags = flags;
    if (!isfinite(st.k3_mean)) st.flags |= TIM_SEQ_K3_OVERFLOW;
    if (flags & TIM_SEQ_NONFINITE) set_status(status, TIM_ERR_NONFINITE);
  }
  out[j] = st;
}

cudaError_t launch_seg_compare(const float* A, const float* B, const float* C,
                               const int64_t* offs, int n_seq, const uint8_t* mask, int64_t T,
                               float tis_cap, tim_seq_stats* out, float* tis_w, int* status,
                               cudaStream_t stream) {
  const double cap = static_cast<double>(tis_cap);
  const double ln_cap = std::log(cap);
  const bool vec = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                     reinterpret_cast<uintptr_t>(C)) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(mask) & 3u) == 0;
  if (vec)
    seg_compare_kernel<true><<<n_seq, kCmpThreads, 0, stream>>>(A, B, C, offs, mask, T, cap,
                                                                ln_cap, out, tis_w, status);
  else
    seg_compare_kernel<false><<<n_seq, kCmpThreads, 0, stream>>>(A, B, C, offs, mask, T, cap,
                                                                 ln_cap, out, tis_w, status);
  return cudaGetLastError();
}

}  // namespace tim
