// Three-way score comparison: a segmented reduction over sequences.
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
// Work split: sequence j is cut into P_j contiguous parts, P_j taken from the
// sequence's own length (so its statistics do not depend on the batch it comes
// in); CTA (j, p) reduces part p to a 256-byte
// partial, and the last CTA of sequence j to finish (an atomic ticket) merges
// the P partials in part order and writes the sequence's statistics.  Inside a
// CTA each thread owns a 4-token vector (128-bit loads of each score array when
// the arrays are 16-byte aligned) and walks its tokens in order; runs of
// differing tokens are combined with the ordered monoid
//   (n, ndiff, first, prefix_run, suffix_run, best_run)
// through a warp shuffle tree (lane i with lane i+o, o = 1, 2, 4, 8, 16) and
// then across warps in warp order.  Counts, first positions, runs and maxima
// are exact; the fp64 sums are taken in a fixed order.
#include <cmath>
#include <cstring>

#include "tim_common.cuh"

namespace tim {

constexpr int kCmpThreads = 64;
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

// One part's reduction (256 bytes, written by CTA (j, p) to the workspace).
// v[]: sgn[3], abs[3], max[3], k3, tis.
struct alignas(16) CmpPart {
  Runs<long long> runs[3];
  double v[11];
  long long clipped;
  int flags;
  int pad;
  int pad2[2];
};
static_assert(sizeof(CmpPart) == 256, "compare partial is 256 bytes");

// Compare workspace: status word | per-sequence tickets int32 [S] | part bases
// int32 [S + 1] | parts [sum of P_j] (at most seq_parts_bound(T, S)).
struct CmpLayout {
  size_t cnt_off, base_off, part_off, total;
};
__host__ inline CmpLayout compare_layout(int64_t T, int n_seq) {
  CmpLayout L;
  L.cnt_off = 256;
  L.base_off = align_up(L.cnt_off + static_cast<size_t>(n_seq) * 4, 256);
  L.part_off = align_up(L.base_off + static_cast<size_t>(n_seq + 1) * 4, 256);
  L.total = align_up(L.part_off + static_cast<size_t>(seq_parts_bound(T, n_seq)) *
                                      sizeof(CmpPart),
                     1024);
  return L;
}

// base[j] = sum of P_i for i < j, base[n_seq] = total; one block, each thread a
// contiguous run of sequences, then a block-wide exclusive scan of the run sums.
// It also zeroes the call's per-sequence tickets (cnt, when given), so they
// start at zero whatever an earlier call of another shape left in the workspace.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
    seq_partition_kernel(const int64_t* __restrict__ offs, int n_seq, int64_t T,
                         int* __restrict__ base, int* __restrict__ cnt) {
  __shared__ int s_warp[kScanThreads / 32];
  pdl_launch_dependents();  // the compare / diagnostics kernel may launch now
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n_seq + kScanThreads - 1) / kScanThreads;
  const int j0 = tid * per;
  const int j1 = j0 + per < n_seq ? j0 + per : n_seq;
  int sum = 0;
  for (int j = j0; j < j1; ++j) sum += seq_parts(offs[j], offs[j + 1], T);
  int incl = sum;  // inclusive scan within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += u;
    }
    s_warp[lane] = w;  // inclusive prefix of the warp sums
  }
  __syncthreads();
  int run = incl - sum + (warp > 0 ? s_warp[warp - 1] : 0);  // exclusive prefix
  for (int j = j0; j < j1; ++j) {
    base[j] = run;
    run += seq_parts(offs[j], offs[j + 1], T);
    if (cnt != nullptr) cnt[j] = 0;
  }
  if (tid == kScanThreads - 1) base[n_seq] = s_warp[31];
}

cudaError_t launch_seq_partition(const int64_t* offs, int n_seq, int64_t T, int* base, int* cnt,
                                 cudaStream_t stream) {
  seq_partition_kernel<<<1, kScanThreads, 0, stream>>>(offs, n_seq, T, base, cnt);
  return cudaGetLastError();
}

struct Acc {
  double v[11];
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
    acc.v[p] += x[p];
    acc.v[3 + p] += fabs(x[p]);
    acc.v[6 + p] = fmax(acc.v[6 + p], fabs(x[p]));
  }
  const double d = dc - da;
  acc.v[9] += expm1(d) - d;
  double w;
  if (d > ln_cap) {
    w = cap;
    acc.clipped += 1;
  } else {
    w = exp(d);
  }
  acc.v[10] += w;
  if (tis_w != nullptr) tis_w[t] = static_cast<float>(w);
}

__device__ __forceinline__ bool is_max_slot(int i) { return i >= 6 && i < 9; }

template <bool kVec>
__global__ void __launch_bounds__(kCmpThreads)
    seg_compare_kernel(const float* __restrict__ A, const float* __restrict__ B,
                       const float* __restrict__ C, const int64_t* __restrict__ offs,
                       const uint8_t* __restrict__ mask, int64_t T, int n_seq,
                       const int* __restrict__ base, double cap, double ln_cap,
                       tim_seq_stats* __restrict__ out, float* __restrict__ tis_w, int* status,
                       int* cnt, CmpPart* parts) {
  __shared__ Runs<int> s_runs[kCmpWarps][3];
  __shared__ double s_red[kCmpWarps][11];
  __shared__ long long s_clip[kCmpWarps];
  __shared__ int s_flags[kCmpWarps];
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;  // global part index
  pdl_wait();  // the partition kernel's bases and zeroed tickets
  if (b >= __ldcg(base + n_seq)) return;
  const int j = part_sequence(base, n_seq, b);
  const int p = b - __ldcg(base + j);
  const int P = __ldcg(base + j + 1) - __ldcg(base + j);
  const int64_t s = offs[j], e = offs[j + 1];
  if (!(s >= 0 && s <= e && e <= T)) {
    if (tid == 0 && p == 0) {
      tim_seq_stats st;
      memset(&st, 0, sizeof(st));
      for (int q = 0; q < 3; ++q) st.pair[q].first_div = -1;
      st.flags = TIM_SEQ_BAD_OFFSETS;
      out[j] = st;
      set_status(status, TIM_ERR_INVALID_ARG);
    }
    return;
  }
  const int64_t len = e - s;
  const int64_t ps = s + len * p / P, pe = s + len * (p + 1) / P;   // this CTA's part

  Acc acc;
#pragma unroll
  for (int i = 0; i < 11; ++i) acc.v[i] = 0.0;
  acc.clipped = 0;
  acc.flags = 0;
  Runs<long long> total[3] = {runs_identity<long long>(), runs_identity<long long>(),
                              runs_identity<long long>()};

  const int64_t vbeg = ps >> 2, vend = (pe + 3) >> 2;
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
          const bool in = (t >= ps && t < pe);
          av[k] = in ? __ldg(A + t) : 0.f;
          bv[k] = in ? __ldg(B + t) : 0.f;
          cv[k] = in ? __ldg(C + t) : 0.f;
          mv[k] = in ? __ldg(mask + t) : 0;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t t = t0 + k;
        if (t < ps || t >= pe) continue;
        if (mv[k] > 1) acc.flags |= TIM_SEQ_BAD_MASK;
        if (mv[k] != 1) {
          if (tis_w != nullptr) tis_w[t] = 0.f;
          continue;
        }
        token(acc, runs, av[k], bv[k], cv[k], cap, ln_cap, tis_w, t);
      }
    }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      runs[q] = warp_runs_reduce(runs[q], lane);
      if (lane == 0) s_runs[warp][q] = runs[q];
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        Runs<int> chunk = runs_identity<int>();
        for (int w = 0; w < kCmpWarps; ++w) chunk = runs_combine(chunk, s_runs[w][q]);
        total[q] = runs_combine(total[q], chunk);
      }
    }
    __syncthreads();
  }

  // fixed-order block reduction of the per-thread accumulators
  double v[11];
#pragma unroll
  for (int i = 0; i < 11; ++i) v[i] = acc.v[i];
  long long clip = acc.clipped;
  int flags = acc.flags;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int i = 0; i < 11; ++i) {
      const double other = __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
      v[i] = is_max_slot(i) ? fmax(v[i], other) : v[i] + other;
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
  if (tid == 0) {
    CmpPart part;
    memset(&part, 0, sizeof(part));
    for (int i = 0; i < 11; ++i) {
      double r = s_red[0][i];
      for (int w = 1; w < kCmpWarps; ++w) r = is_max_slot(i) ? fmax(r, s_red[w][i]) : r + s_red[w][i];
      part.v[i] = r;
    }
    for (int w = 0; w < kCmpWarps; ++w) {
      part.clipped += s_clip[w];
      part.flags |= s_flags[w];
    }
    for (int q = 0; q < 3; ++q) part.runs[q] = total[q];
    parts[b] = part;
    __threadfence();
    const int ticket = atomicAdd(&cnt[j], 1);
    s_last = (ticket == P - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last || warp != 0) return;

  // last CTA of sequence j: warp 0 merges the P partials in part order.  Lane l
  // folds the contiguous block of parts [l*per, (l+1)*per) in order (its loads
  // all in flight together), then an ordered tree across lanes combines lane l
  // (left) with lane l + off (right), so the run statistics keep the sequence
  // order.
  __threadfence();
  const CmpPart* pj = parts + __ldcg(base + j);
  Runs<long long> R[3] = {runs_identity<long long>(), runs_identity<long long>(),
                          runs_identity<long long>()};
  double tot[11];
  for (int i = 0; i < 11; ++i) tot[i] = 0.0;
  long long clipped = 0;
  int fl = 0;
  const int per = (P + 31) / 32;
  const int q0 = lane * per;
  const int q1 = q0 + per < P ? q0 + per : P;
  for (int q = q0; q < q1; ++q) {
    const CmpPart* pp = pj + q;
    for (int r = 0; r < 3; ++r) {
      Runs<long long> x;
      x.n = __ldcg(&pp->runs[r].n);
      x.ndiff = __ldcg(&pp->runs[r].ndiff);
      x.first = __ldcg(&pp->runs[r].first);
      x.pre = __ldcg(&pp->runs[r].pre);
      x.suf = __ldcg(&pp->runs[r].suf);
      x.best = __ldcg(&pp->runs[r].best);
      R[r] = runs_combine(R[r], x);
    }
    for (int i = 0; i < 11; ++i) {
      const double x = __ldcg(&pp->v[i]);
      tot[i] = is_max_slot(i) ? fmax(tot[i], x) : tot[i] + x;
    }
    clipped += __ldcg(&pp->clipped);
    fl |= __ldcg(&pp->flags);
  }
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    Runs<long long> o[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      o[r].n = __shfl_down_sync(0xFFFFFFFFu, R[r].n, off);
      o[r].ndiff = __shfl_down_sync(0xFFFFFFFFu, R[r].ndiff, off);
      o[r].first = __shfl_down_sync(0xFFFFFFFFu, R[r].first, off);
      o[r].pre = __shfl_down_sync(0xFFFFFFFFu, R[r].pre, off);
      o[r].suf = __shfl_down_sync(0xFFFFFFFFu, R[r].suf, off);
      o[r].best = __shfl_down_sync(0xFFFFFFFFu, R[r].best, off);
    }
    double ot[11];
#pragma unroll
    for (int i = 0; i < 11; ++i) ot[i] = __shfl_down_sync(0xFFFFFFFFu, tot[i], off);
    const long long oc = __shfl_down_sync(0xFFFFFFFFu, clipped, off);
    const int of = __shfl_down_sync(0xFFFFFFFFu, fl, off);
    if ((lane & (2 * off - 1)) == 0 && lane + off < 32) {
#pragma unroll
      for (int r = 0; r < 3; ++r) R[r] = runs_combine(R[r], o[r]);
#pragma unroll
      for (int i = 0; i < 11; ++i) tot[i] = is_max_slot(i) ? fmax(tot[i], ot[i]) : tot[i] + ot[i];
      clipped += oc;
      fl |= of;
    }
  }
  if (lane != 0) return;

  tim_seq_stats st;
  memset(&st, 0, sizeof(st));
  for (int q = 0; q < 3; ++q) st.pair[q].first_div = -1;
  const long long n = R[0].n;
  if (fl & TIM_SEQ_BAD_MASK) {
    st.flags = TIM_SEQ_BAD_MASK;
    set_status(status, TIM_ERR_BAD_MASK);
  } else if (n == 0) {
    st.flags = TIM_SEQ_EMPTY;
    set_status(status, TIM_ERR_EMPTY_SEQUENCE);
  } else {
    const double dn = static_cast<double>(n);
    st.n_valid = n;
    for (int q = 0; q < 3; ++q) {
      st.pair[q].mismatch_count = R[q].ndiff;
      st.pair[q].first_div = R[q].first;
      st.pair[q].longest_run = R[q].best;
      st.pair[q].max_abs_diff = tot[6 + q];
      st.pair[q].signed_mean = tot[q] / dn;
      st.pair[q].mae = tot[3 + q] / dn;
    }
    st.mean_log_ratio = -tot[2] / dn;
    st.mean_weight_move = -tot[1] / dn;
    st.mean_same_version = -tot[0] / dn;
    st.k3_mean = tot[9] / dn;
    st.tis_mean = tot[10] / dn;
    st.tis_clipped = clipped;
    st.flags = fl;
    if (!isfinite(st.k3_mean)) st.flags |= TIM_SEQ_K3_OVERFLOW;
    if (fl & TIM_SEQ_NONFINITE) set_status(status, TIM_ERR_NONFINITE);
  }
  out[j] = st;
}

size_t compare_workspace_bytes(int64_t T, int n_seq) { return compare_layout(T, n_seq).total; }

cudaError_t launch_seg_compare(const float* A, const float* B, const float* C,
                               const int64_t* offs, int n_seq, const uint8_t* mask, int64_t T,
                               float tis_cap, tim_seq_stats* out, float* tis_w, void* workspace,
                               cudaStream_t stream) {
  const double cap = static_cast<double>(tis_cap);
  const double ln_cap = std::log(cap);
  const CmpLayout L = compare_layout(T, n_seq);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  int* cnt = reinterpret_cast<int*>(ws + L.cnt_off);
  int* base = reinterpret_cast<int*>(ws + L.base_off);
  CmpPart* parts = reinterpret_cast<CmpPart*>(ws + L.part_off);
  cudaError_t e = launch_seq_partition(offs, n_seq, T, base, cnt, stream);
  if (e != cudaSuccess) return e;
  const bool vec = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                     reinterpret_cast<uintptr_t>(C)) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(mask) & 3u) == 0;
  // Programmatic dependent launch: the compare kernel launches while the
  // partition kernel runs and waits for its results (griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(seq_parts_bound(T, n_seq)));
  cfg.blockDim = dim3(kCmpThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (vec)
    return cudaLaunchKernelEx(&cfg, seg_compare_kernel<true>, A, B, C, offs, mask, T, n_seq,
                              static_cast<const int*>(base), cap, ln_cap, out, tis_w, status, cnt,
                              parts);
  return cudaLaunchKernelEx(&cfg, seg_compare_kernel<false>, A, B, C, offs, mask, T, n_seq,
                            static_cast<const int*>(base), cap, ln_cap, out, tis_w, status, cnt,
                            parts);
}

}  // namespace tim
