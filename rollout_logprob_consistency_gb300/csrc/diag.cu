// Extended per-sequence mismatch diagnostics, one CTA per sequence.
//
// Same roles and masking as the three-way compare (A generation, B replay,
// C trainer; pairs A-B, B-C, A-C; active tokens only; d = C - A).  Per sequence:
//  - |left - right| p50 / p95 / p99 per pair ("Diagnosing Training Inference
//    Mismatch in LLM Reinforcement Learning", 5. practical indicators; the
//    p95 / p99 of the compare summary of "Debugging Logprob Mismatches in LLM
//    Reinforcement Learning", Case 1), linear interpolation between order
//    statistics: h = (n-1) q, Q = x[floor h] + (h - floor h)(x[floor h + 1] - x[floor h]);
//  - probability MAE per pair, mean |exp(left) - exp(right)| ("Fault
//    localization and mismatch bisect", Metric measurement basis);
//  - top-1 flips per pair (practical indicators: top-1 token flip rate);
//  - sum d, k1 sum = -sum d, k3 sum = sum(expm1(d) - d) (sequence rejection by
//    sum_t K1 / K3 of the correction ratio, "Diagnosing ...", 3. TIS);
//  - sequence TIS min(exp(sum d), cap) (same section);
//  - ratio error mean |exp(d) - 1| (practical indicators: PPO ratio error);
//  - MIS: w 1[lo <= w <= hi], w = exp(d) ("Rollout-Training Mismatch in LLM RL",
//    section 2.1); mean w^2 = mean exp(2d) (same page, section 5.3).
//
// Sums: each thread accumulates its strided tokens in order, then a fixed
// xor-butterfly and warp-order reduction (deterministic).  Quantiles: the
// sequence's |left - right| values of active tokens are gathered into shared
// memory (any order), padded with +inf to a power of two and bitonic-sorted;
// the order statistics are exact, the interpolation is the formula above.
// Sequences with more than kQuantMax active tokens skip the quantiles (flag).
#include <cmath>
#include <cstring>

#include "tim_common.cuh"

namespace tim {

constexpr int kDiagThreads = 512;
constexpr int kDiagWarps = kDiagThreads / 32;
constexpr int kQuantMax = TIM_DIAG_QUANTILE_MAX_TOKENS;
constexpr size_t kDiagSmemBytes = static_cast<size_t>(kQuantMax) * sizeof(double);

// per-thread sums: prob[3], dsum, k3, rerr, mis, w2
constexpr int kDiagSums = 8;
// per-thread counts: n, kept, flips[3]
constexpr int kDiagCounts = 5;

__device__ __forceinline__ double pair_abs(int p, double a, double b, double c) {
  return p == 0 ? fabs(a - b) : (p == 1 ? fabs(b - c) : fabs(a - c));
}

__global__ void __launch_bounds__(kDiagThreads)
    seg_diag_kernel(const float* __restrict__ A, const float* __restrict__ B,
                    const float* __restrict__ C, const int32_t* __restrict__ tA,
                    const int32_t* __restrict__ tB, const int32_t* __restrict__ tC,
                    const int64_t* __restrict__ offs, const uint8_t* __restrict__ mask,
                    int64_t T, double cap, double ln_cap, double ln_lo, double ln_hi,
                    tim_seq_diag* __restrict__ out, int* status) {
  extern __shared__ double buf[];
  __shared__ double s_sum[kDiagWarps][kDiagSums];
  __shared__ long long s_cnt[kDiagWarps][kDiagCounts];
  __shared__ int s_flags[kDiagWarps];
  __shared__ int s_fill;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = blockIdx.x;
  const int64_t s = offs[j], e = offs[j + 1];
  tim_seq_diag st;
  if (!(s >= 0 && s <= e && e <= T)) {
    if (tid == 0) {
      memset(&st, 0, sizeof(st));
      for (int p = 0; p < 3; ++p) st.top1_flips[p] = -1;
      st.flags = TIM_SEQ_BAD_OFFSETS;
      out[j] = st;
      set_status(status, TIM_ERR_INVALID_ARG);
    }
    return;
  }

  double sum[kDiagSums];
  long long cnt[kDiagCounts];
#pragma unroll
  for (int i = 0; i < kDiagSums; ++i) sum[i] = 0.0;
#pragma unroll
  for (int i = 0; i < kDiagCounts; ++i) cnt[i] = 0;
  int flags = 0;

  for (int64_t t = s + tid; t < e; t += kDiagThreads) {
    const uint8_t m = __ldg(mask + t);
    if (m > 1) flags |= TIM_SEQ_BAD_MASK;
    if (m != 1) continue;
    const float a = __ldg(A + t), b = __ldg(B + t), c = __ldg(C + t);
    if (!(isfinite(a) && isfinite(b) && isfinite(c))) flags |= TIM_SEQ_NONFINITE;
    const double da = a, db = b, dc = c;
    const double ea = exp(da), eb = exp(db), ec = exp(dc);
    sum[0] += fabs(ea - eb);
    sum[1] += fabs(eb - ec);
    sum[2] += fabs(ea - ec);
    const double d = dc - da;
    const double em1 = expm1(d);
    sum[3] += d;
    sum[4] += em1 - d;
    sum[5] += fabs(em1);
    if (d >= ln_lo && d <= ln_hi) {
      sum[6] += exp(d);
      cnt[1] += 1;
    }
    sum[7] += exp(2.0 * d);
    cnt[0] += 1;
    if (tA != nullptr && tB != nullptr) cnt[2] += (__ldg(tA + t) != __ldg(tB + t)) ? 1 : 0;
    if (tB != nullptr && tC != nullptr) cnt[3] += (__ldg(tB + t) != __ldg(tC + t)) ? 1 : 0;
    if (tA != nullptr && tC != nullptr) cnt[4] += (__ldg(tA + t) != __ldg(tC + t)) ? 1 : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int i = 0; i < kDiagSums; ++i) sum[i] += __shfl_xor_sync(0xFFFFFFFFu, sum[i], o);
#pragma unroll
    for (int i = 0; i < kDiagCounts; ++i) cnt[i] += __shfl_xor_sync(0xFFFFFFFFu, cnt[i], o);
    flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, o);
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kDiagSums; ++i) s_sum[warp][i] = sum[i];
#pragma unroll
    for (int i = 0; i < kDiagCounts; ++i) s_cnt[warp][i] = cnt[i];
    s_flags[warp] = flags;
  }
  __syncthreads();
  // every thread folds the warp partials in warp order (same bits everywhere)
  double S[kDiagSums];
  long long N[kDiagCounts];
  int F = 0;
#pragma unroll
  for (int i = 0; i < kDiagSums; ++i) S[i] = 0.0;
#pragma unroll
  for (int i = 0; i < kDiagCounts; ++i) N[i] = 0;
  for (int w = 0; w < kDiagWarps; ++w) {
#pragma unroll
    for (int i = 0; i < kDiagSums; ++i) S[i] += s_sum[w][i];
#pragma unroll
    for (int i = 0; i < kDiagCounts; ++i) N[i] += s_cnt[w][i];
    F |= s_flags[w];
  }
  const long long n = N[0];
  const bool valid = !(F & TIM_SEQ_BAD_MASK) && n > 0;

  double q50[3] = {0, 0, 0}, q95[3] = {0, 0, 0}, q99[3] = {0, 0, 0};
  const bool do_q = valid && n <= kQuantMax;
  if (do_q) {
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int p = 0; p < 3; ++p) {
      if (tid == 0) s_fill = 0;
      __syncthreads();
      for (int64_t t = s + tid; t < e; t += kDiagThreads) {
        if (__ldg(mask + t) != 1) continue;
        const double a = __ldg(A + t), b = __ldg(B + t), c = __ldg(C + t);
        const int slot = atomicAdd(&s_fill, 1);
        if (slot < kQuantMax) buf[slot] = pair_abs(p, a, b, c);
      }
      __syncthreads();
      for (int i = static_cast<int>(n) + tid; i < n2; i += kDiagThreads) buf[i] = INFINITY;
      __syncthreads();
      for (int k = 2; k <= n2; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
          for (int i = tid; i < n2; i += kDiagThreads) {
            const int ixj = i ^ jj;
            if (ixj > i) {
              const double x = buf[i], y = buf[ixj];
              const bool up = (i & k) == 0;
              if ((x > y) == up) {
                buf[i] = y;
                buf[ixj] = x;
              }
            }
          }
          __syncthreads();
        }
      }
      if (tid == 0) {
        const double qs[3] = {0.5, 0.95, 0.99};
        double r[3];
        for (int qi = 0; qi < 3; ++qi) {
          const double h = static_cast<double>(n - 1) * qs[qi];
          const double fl = floor(h);
          const long long lo = static_cast<long long>(fl);
          const long long hi = lo + 1 < n ? lo + 1 : n - 1;
          r[qi] = buf[lo] + (h - fl) * (buf[hi] - buf[lo]);
        }
        q50[p] = r[0];
        q95[p] = r[1];
        q99[p] = r[2];
      }
      __syncthreads();
    }
  }
  if (tid != 0) return;

  memset(&st, 0, sizeof(st));
  for (int p = 0; p < 3; ++p) st.top1_flips[p] = -1;
  if (F & TIM_SEQ_BAD_MASK) {
    st.flags = TIM_SEQ_BAD_MASK;
    set_status(status, TIM_ERR_BAD_MASK);
  } else if (n == 0) {
    st.flags = TIM_SEQ_EMPTY;
    set_status(status, TIM_ERR_EMPTY_SEQUENCE);
  } else {
    const double dn = static_cast<double>(n);
    st.n_valid = n;
    for (int p = 0; p < 3; ++p) {
      st.abs_q50[p] = do_q ? q50[p] : NAN;
      st.abs_q95[p] = do_q ? q95[p] : NAN;
      st.abs_q99[p] = do_q ? q99[p] : NAN;
      st.prob_mae[p] = S[p] / dn;
    }
    if (tA != nullptr && tB != nullptr) st.top1_flips[0] = N[2];
    if (tB != nullptr && tC != nullptr) st.top1_flips[1] = N[3];
    if (tA != nullptr && tC != nullptr) st.top1_flips[2] = N[4];
    st.log_ratio_sum = S[3];
    st.k1_sum = -S[3];
    st.k3_sum = S[4];
    st.seq_tis = S[3] > ln_cap ? cap : exp(S[3]);
    st.ratio_err_mean = S[5] / dn;
    st.mis_mean = S[6] / dn;
    st.mis_kept = N[1];
    st.w2_mean = S[7] / dn;
    st.flags = F;
    if (!do_q) st.flags |= TIM_SEQ_QUANTILE_SKIPPED;
    if (!isfinite(st.k3_sum)) st.flags |= TIM_SEQ_K3_OVERFLOW;
    if (F & TIM_SEQ_NONFINITE) set_status(status, TIM_ERR_NONFINITE);
  }
  out[j] = st;
}

cudaError_t launch_seg_diag(const float* A, const float* B, const float* C, const int32_t* tA,
                            const int32_t* tB, const int32_t* tC, const int64_t* offs, int n_seq,
                            const uint8_t* mask, int64_t T, float tis_cap, float mis_lo,
                            float mis_hi, tim_seq_diag* out, int* status, cudaStream_t stream) {
  const double cap = static_cast<double>(tis_cap);
  cudaError_t err = cudaFuncSetAttribute(seg_diag_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kDiagSmemBytes));
  if (err != cudaSuccess) return err;
  seg_diag_kernel<<<n_seq, kDiagThreads, kDiagSmemBytes, stream>>>(
      A, B, C, tA, tB, tC, offs, mask, T, cap, std::log(cap),
      std::log(static_cast<double>(mis_lo)), std::log(static_cast<double>(mis_hi)), out, status);
  return cudaGetLastError();
}

}  // namespace tim
