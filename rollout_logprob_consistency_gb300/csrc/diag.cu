// Extended per-sequence mismatch diagnostics.
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
// Work split, one launch: each sequence is cut into P_j contiguous parts with
// P_j from its own length (as in the compare kernel, so a sequence's results do
// not depend on the batch); a part CTA accumulates its tokens per thread in
// order, then a fixed xor-butterfly and warp-order fold, writes one partial
// record and draws a ticket on the sequence's counter, and the CTA with the last
// ticket folds the P partials in part order (deterministic) into every field but
// the quantiles.  Three more CTAs per sequence, independent of the parts, gather
// one pair's |left - right| values of the active tokens into shared memory (any
// order) as 64-bit keys (the bit patterns of non-negative doubles order like
// the values, so selection is integer work) and find the order statistics the
// interpolation needs by a radix select; they are exact, and the interpolation
// is the formula above.  A sequence with more active tokens than the shared
// key buffer holds (kQuantMax) keeps the keys past the first kQuantMax in a
// workspace region (8 bytes per token and pair) and runs the same select over
// both.
#include <cmath>
#include <cstring>

#include "tim_common.cuh"

namespace tim {

constexpr int kDiagThreads = 512;  // every CTA: quantile selects and per-token parts
constexpr int kDiagWarps = kDiagThreads / 32;
constexpr int kQuantMax = 16384;  // keys a quantile CTA holds in shared memory
constexpr size_t kDiagSmemBytes = static_cast<size_t>(kQuantMax) * sizeof(unsigned long long);

// per-part sums: prob[3], dsum, k3, rerr, mis, w2
constexpr int kDiagSums = 8;
// per-part counts: n, kept, flips[3]
constexpr int kDiagCounts = 5;

struct DiagPart {
  double sum[kDiagSums];
  long long cnt[kDiagCounts];
  int flags;
  int pad;
};
static_assert(sizeof(DiagPart) % sizeof(unsigned long long) == 0, "DiagPart is staged in 8-byte words");
static_assert(static_cast<size_t>(kSeqMaxParts) * sizeof(DiagPart) <= kDiagSmemBytes,
              "a sequence's partials fit the shared key buffer");

cudaError_t launch_seq_partition(const int64_t* offs, int n_seq, int64_t T, int* base, int* cnt,
                                 cudaStream_t stream);

// |a - b| of two floats, as the bit pattern of the double (double)a - (double)b
// rounded to nearest.  When the fp32 difference is exact (TwoSum's error term is
// zero, which Sterbenz's lemma guarantees for operands within a factor of two)
// and normal or zero, the double is that float widened, built with integer
// operations; otherwise the fp64 subtraction runs.  GB300's fp64 pipe is narrow,
// and every active token of a sequence passes through here.
__device__ __forceinline__ unsigned long long abs_diff_key(float a, float b) {
  const float s = __fsub_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  const float err = __fadd_rn(__fsub_rn(a, av), __fsub_rn(-b, bv));  // s + err = a - b
  const uint32_t u = __float_as_uint(s) & 0x7FFFFFFFu;
  const uint32_t ex = u >> 23;
  if (err == 0.f) {
    if (u == 0u) return 0ull;
    if (ex != 0u && ex != 255u)  // rebias the exponent, widen the fraction
      return (static_cast<unsigned long long>(ex + (1023u - 127u)) << 52) |
             (static_cast<unsigned long long>(u & 0x7FFFFFu) << 29);
  }
  return static_cast<unsigned long long>(
      __double_as_longlong(fabs(static_cast<double>(a) - static_cast<double>(b))));
}

__device__ __forceinline__ unsigned long long warp_or_u64(unsigned long long v) {
  const unsigned lo = __reduce_or_sync(0xFFFFFFFFu, static_cast<unsigned>(v));
  const unsigned hi = __reduce_or_sync(0xFFFFFFFFu, static_cast<unsigned>(v >> 32));
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

__device__ __forceinline__ unsigned long long warp_and_u64(unsigned long long v) {
  const unsigned lo = __reduce_and_sync(0xFFFFFFFFu, static_cast<unsigned>(v));
  const unsigned hi = __reduce_and_sync(0xFFFFFFFFu, static_cast<unsigned>(v >> 32));
  return (static_cast<unsigned long long>(hi) << 32) | lo;
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w < v ? w : v;
  }
  return v;
}

// Warp totals of 8 per-lane doubles by recursive halving: at xor offsets 16, 8
// and 4 a lane keeps half of its remaining sums (adding the partner's) and
// hands the other half over, then offsets 2 and 1 finish the one it kept.
// Each level adds the same two subtrees as a full xor butterfly, so every
// total has the butterfly's bits, for 9 additions a lane instead of 40.
// Returns the total of sum kind 4 (lane & 16 ? 1 : 0) + 2 (lane & 8 ? 1 : 0) +
// (lane & 4 ? 1 : 0).
__device__ __forceinline__ double warp_sum8_halving(const double (&v)[8], int lane) {
  double w4[4], w2[2];
  const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0, h4 = (lane & 4) != 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const double give = h16 ? v[i] : v[4 + i];
    const double keep = h16 ? v[4 + i] : v[i];
    w4[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const double give = h8 ? w4[i] : w4[2 + i];
    const double keep = h8 ? w4[2 + i] : w4[i];
    w2[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 8);
  }
  double z = (h4 ? w2[1] : w2[0]) + __shfl_xor_sync(0xFFFFFFFFu, h4 ? w2[0] : w2[1], 4);
  z += __shfl_xor_sync(0xFFFFFFFFu, z, 2);
  z += __shfl_xor_sync(0xFFFFFFFFu, z, 1);
  return z;
}

__device__ __forceinline__ bool offsets_ok(int64_t s, int64_t e, int64_t T) {
  return s >= 0 && s <= e && e <= T;
}

// Every field of sequence j's record but the quantiles, from its P partials
// (staged in shared memory) folded in part order by one warp: lane i < 8 sums
// partial field i, lanes 8-12 the counts, lane 13 ORs the flags; the quotients
// and the exponential then run on separate lanes.
__device__ void diag_fold(int j, bool ok_offs, const int32_t* __restrict__ tA,
                          const int32_t* __restrict__ tB, const int32_t* __restrict__ tC,
                          double cap, double ln_cap, const DiagPart* __restrict__ pj, int P,
                          tim_seq_diag* __restrict__ o, int* status) {
  const int lane = threadIdx.x & 31;
  if (!ok_offs) {
    if (lane == 0) {
      tim_seq_diag st;
      memset(&st, 0, sizeof(st));
      for (int p = 0; p < 3; ++p) st.top1_flips[p] = -1;
      st.flags = TIM_SEQ_BAD_OFFSETS;
      *o = st;
      set_status(status, TIM_ERR_INVALID_ARG);
    }
    return;
  }
  double acc = 0.0;
  long long cacc = 0;
  int facc = 0;
  for (int q = 0; q < P; ++q) {  // part order
    const DiagPart& r = pj[q];
    if (lane < kDiagSums) acc += r.sum[lane];
    else if (lane < kDiagSums + kDiagCounts) cacc += r.cnt[lane - kDiagSums];
    else if (lane == kDiagSums + kDiagCounts) facc |= r.flags;
  }
  double S[kDiagSums];
  long long N[kDiagCounts];
#pragma unroll
  for (int i = 0; i < kDiagSums; ++i) S[i] = __shfl_sync(0xFFFFFFFFu, acc, i);
#pragma unroll
  for (int i = 0; i < kDiagCounts; ++i) N[i] = __shfl_sync(0xFFFFFFFFu, cacc, kDiagSums + i);
  const int F = __shfl_sync(0xFFFFFFFFu, facc, kDiagSums + kDiagCounts);
  const long long n = N[0];
  const bool ok = !(F & TIM_SEQ_BAD_MASK) && n > 0;
  double v = 0.0;  // lane 0-2: probability MAE; 3: ratio error; 4: MIS; 5: w^2; 6: sequence TIS
  if (ok && lane < 7) {
    const double dn = static_cast<double>(n);
    if (lane < 3) v = acc / dn;  // lane i < 8 holds S[i]
    else if (lane == 3) v = S[5] / dn;
    else if (lane == 4) v = S[6] / dn;
    else if (lane == 5) v = S[7] / dn;
    else v = S[3] > ln_cap ? cap : exp(S[3]);
  }
  double q[7];
#pragma unroll
  for (int i = 0; i < 7; ++i) q[i] = __shfl_sync(0xFFFFFFFFu, v, i);
  if (lane != 0) return;
  // every field except the quantiles (written by the quantile CTAs)
  o->reserved = 0;
  for (int p = 0; p < 3; ++p) {
    o->prob_mae[p] = 0.0;
    o->top1_flips[p] = -1;
  }
  o->n_valid = 0;
  o->log_ratio_sum = o->k1_sum = o->k3_sum = o->seq_tis = 0.0;
  o->ratio_err_mean = o->mis_mean = o->w2_mean = 0.0;
  o->mis_kept = 0;
  if (F & TIM_SEQ_BAD_MASK) {
    o->flags = TIM_SEQ_BAD_MASK;
    set_status(status, TIM_ERR_BAD_MASK);
  } else if (n == 0) {
    o->flags = TIM_SEQ_EMPTY;
    set_status(status, TIM_ERR_EMPTY_SEQUENCE);
  } else {
    o->n_valid = n;
    for (int p = 0; p < 3; ++p) o->prob_mae[p] = q[p];
    if (tA != nullptr && tB != nullptr) o->top1_flips[0] = N[2];
    if (tB != nullptr && tC != nullptr) o->top1_flips[1] = N[3];
    if (tA != nullptr && tC != nullptr) o->top1_flips[2] = N[4];
    o->log_ratio_sum = S[3];
    o->k1_sum = -S[3];
    o->k3_sum = S[4];
    o->seq_tis = q[6];
    o->ratio_err_mean = q[3];
    o->mis_mean = q[4];
    o->mis_kept = N[1];
    o->w2_mean = q[5];
    int flags = F;
    if (!isfinite(S[4])) flags |= TIM_SEQ_K3_OVERFLOW;
    o->flags = flags;
    if (F & TIM_SEQ_NONFINITE) set_status(status, TIM_ERR_NONFINITE);
  }
}

// One part of a sequence: its tokens' sums, then a ticket on the sequence's
// counter; the CTA that draws the last ticket folds the sequence's parts.
__device__ void diag_part(int b, unsigned long long* __restrict__ stage,
                          const float* __restrict__ A, const float* __restrict__ B,
                          const float* __restrict__ C, const int32_t* __restrict__ tA,
                          const int32_t* __restrict__ tB, const int32_t* __restrict__ tC,
                          const int64_t* __restrict__ offs, const uint8_t* __restrict__ mask,
                          int64_t T, int n_seq, const int* __restrict__ base, double ln_lo,
                          double ln_hi, double cap, double ln_cap, DiagPart* __restrict__ parts,
                          int* __restrict__ cnt_seq, tim_seq_diag* __restrict__ out,
                          int* status) {
  __shared__ double s_sum[kDiagWarps][kDiagSums];
  __shared__ long long s_cnt[kDiagWarps][kDiagCounts];
  __shared__ int s_flags[kDiagWarps];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (b >= __ldcg(base + n_seq)) return;
  const int j = part_sequence(base, n_seq, b);
  const int part = b - __ldcg(base + j);
  const int P = __ldcg(base + j + 1) - __ldcg(base + j);
  const int64_t s = offs[j], e = offs[j + 1];
  const bool ok_offs = offsets_ok(s, e, T);  // bad offsets: one part, no tokens
  const int64_t chunk = ok_offs ? (e - s + P - 1) / P : 0;
  const int64_t t0 = s + static_cast<int64_t>(part) * chunk;
  const int64_t t1 = !ok_offs ? t0 : (t0 + chunk < e ? t0 + chunk : e);

  double sum[kDiagSums];
  long long cnt[kDiagCounts];
#pragma unroll
  for (int i = 0; i < kDiagSums; ++i) sum[i] = 0.0;
#pragma unroll
  for (int i = 0; i < kDiagCounts; ++i) cnt[i] = 0;
  int flags = 0;
  for (int64_t t = t0 + tid; t < t1; t += kDiagThreads) {
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
  // Only warps that held tokens reduce (their butterfly is fp64 work on a
  // narrow pipe); a warp without tokens would only add exact zeros.
  const int64_t n_tok = t1 - t0;
  const int busy_warps =
      n_tok >= static_cast<int64_t>(kDiagThreads) ? kDiagWarps : static_cast<int>((n_tok + 31) / 32);
  static_assert(kDiagSums == 8, "the halving reduction is written for 8 sums");
  if (warp < busy_warps) {
    const double tot = warp_sum8_halving(sum, lane);
    if ((lane & 3) == 0) s_sum[warp][((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)] = tot;
    // counts: at most a few million per warp, exact in 32-bit integer reductions
    long long wc[kDiagCounts];
#pragma unroll
    for (int i = 0; i < kDiagCounts; ++i)
      wc[i] = __reduce_add_sync(0xFFFFFFFFu, static_cast<unsigned>(cnt[i]));
    const int wf = static_cast<int>(__reduce_or_sync(0xFFFFFFFFu, static_cast<unsigned>(flags)));
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kDiagCounts; ++i) s_cnt[warp][i] = wc[i];
      s_flags[warp] = wf;
    }
  }
  __syncthreads();
  if (tid == 0) {
    DiagPart r;
#pragma unroll
    for (int i = 0; i < kDiagSums; ++i) r.sum[i] = 0.0;
#pragma unroll
    for (int i = 0; i < kDiagCounts; ++i) r.cnt[i] = 0;
    r.flags = 0;
    r.pad = 0;
    for (int w = 0; w < busy_warps; ++w) {  // warp order
#pragma unroll
      for (int i = 0; i < kDiagSums; ++i) r.sum[i] += s_sum[w][i];
#pragma unroll
      for (int i = 0; i < kDiagCounts; ++i) r.cnt[i] += s_cnt[w][i];
      r.flags |= s_flags[w];
    }
    parts[b] = r;
    __threadfence();
    s_last = atomicAdd(&cnt_seq[j], 1) == P - 1;
  }
  __syncthreads();
  if (!s_last) return;
  // the last part CTA of sequence j: stage its P partials (written by other
  // CTAs of this launch, so read through L2) and fold them on one warp
  __threadfence();
  constexpr int kWords = static_cast<int>(sizeof(DiagPart) / sizeof(unsigned long long));
  const unsigned long long* src =
      reinterpret_cast<const unsigned long long*>(parts + __ldcg(base + j));
  for (int i = tid; i < P * kWords; i += kDiagThreads) stage[i] = __ldcg(src + i);
  __syncthreads();
  if (warp != 0) return;
  diag_fold(j, ok_offs, tA, tB, tC, cap, ln_cap, reinterpret_cast<const DiagPart*>(stage), P,
            out + j, status);
}

// The active keys of one pair of one sequence, visited by every thread of a
// CTA with a uniform trip count: the first kQuantMax from shared memory, the
// rest (sequences longer than that) from the workspace region the gather wrote
// them to (read through L2: this CTA wrote them during this launch).  Visit
// order is irrelevant to the selection.
struct KeySource {
  const unsigned long long* keys;
  const unsigned long long* spill;
  int n;

  template <class F>
  __device__ __forceinline__ void visit(int tid, F&& f) const {
    const int n_round = (n + kDiagThreads - 1) / kDiagThreads * kDiagThreads;
    const int n_smem = n < kQuantMax ? n : kQuantMax;
#pragma unroll 4
    for (int i = tid; i < n_round; i += kDiagThreads) {
      if (i < n_smem) f(keys[i]);
      else if (i < n) f(__ldcg(spill + (i - kQuantMax)));
    }
  }
};

// Quantiles of pair p of sequence j (one CTA; keys: kQuantMax 64-bit slots in
// shared memory; spill: the workspace region for pair p's keys past those,
// indexed from the sequence's first token).
__device__ void diag_quantiles(int j, int p, unsigned long long* __restrict__ keys,
                               unsigned long long* __restrict__ spill,
                               const float* __restrict__ A, const float* __restrict__ B,
                               const float* __restrict__ C, const int64_t* __restrict__ offs,
                               const uint8_t* __restrict__ mask, int64_t T,
                               tim_seq_diag* __restrict__ out) {
  __shared__ int s_fill, s_bad;
  __shared__ unsigned s_hist[3 * 256];  // radix-select digit counts per target
  __shared__ unsigned long long s_prefix[3], s_mask[3];
  __shared__ unsigned long long s_or[4], s_and[4];  // [q]: target q's candidates; [3]: all keys
  __shared__ unsigned long long s_wmin[kDiagWarps][6];
  __shared__ int s_rem[3], s_cnt[3], s_open[3];
  const int tid = threadIdx.x;
  const int64_t s = offs[j], e = offs[j + 1];
  tim_seq_diag* o = out + j;
  if (!offsets_ok(s, e, T)) return;  // the fold writes the whole record
  if (tid == 0) {
    s_fill = 0;
    s_bad = 0;
  }
  if (tid < 4) {
    s_or[tid] = 0ull;
    s_and[tid] = ~0ull;
  }
  for (int i = tid; i < 3 * 256; i += kDiagThreads) s_hist[i] = 0u;
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5;
  const float* L = p == 1 ? B : A;
  const float* R = p == 0 ? B : C;
  unsigned long long k_or = 0ull, k_and = ~0ull;
  for (int64_t base = s; base < e; base += kDiagThreads) {  // uniform trip count
    const int64_t t = base + tid;
    const uint8_t m = t < e ? __ldg(mask + t) : 0;
    if (m > 1) s_bad = 1;
    const bool act = (m == 1);
    // one shared-memory atomic per warp: the warp's active lanes take consecutive slots
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, act);
    int slot0 = 0;
    if (lane == 0 && bal != 0u) slot0 = atomicAdd(&s_fill, __popc(bal));
    slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
    if (act) {
      const unsigned long long k = abs_diff_key(__ldg(L + t), __ldg(R + t));
      k_or |= k;
      k_and &= k;
      const int slot = slot0 + __popc(bal & ((1u << lane) - 1u));
      if (slot < kQuantMax) keys[slot] = k;
      else spill[s + (slot - kQuantMax)] = k;  // slot < e - s: inside the sequence's range
    }
  }
  k_or = warp_or_u64(k_or);
  k_and = warp_and_u64(k_and);
  if (lane == 0) {
    atomicOr(&s_or[3], k_or);
    atomicAnd(&s_and[3], k_and);
  }
  __syncthreads();
  const int n = s_fill;
  if (s_bad || n == 0) {
    if (tid == 0) {
      o->abs_q50[p] = 0.0;
      o->abs_q95[p] = 0.0;
      o->abs_q99[p] = 0.0;
    }
    return;
  }
  const KeySource src{keys, spill + s, n};
  // The three order statistics by an MSD radix select on the keys' bit
  // patterns.  Target q keeps the key prefix fixed so far (bits [fixed_from,
  // 64)), the rank it still seeks among the keys with that prefix (its
  // candidates) and their count.  Bits every key shares are fixed before the
  // first pass.  A pass histograms the next 8 bits of every candidate of each
  // open target (shared-memory atomics) and takes the OR and AND of the
  // candidates; then warp q either settles target q (the OR equals the AND:
  // every candidate is the same key) or walks its histogram to the digit that
  // holds the rank.  A target also settles when one candidate is left or no
  // bits remain.  Any exact selection on this total order returns the
  // elements a sort would put at those ranks, whatever the gather order.
  const double qs[3] = {0.5, 0.95, 0.99};
  const unsigned long long diff = s_or[3] ^ s_and[3];
  int fixed_from = diff == 0ull ? 0 : 64 - __clzll(static_cast<long long>(diff));
  if (tid < 3) {
    const unsigned long long m0 = fixed_from == 64 ? 0ull : (~0ull << fixed_from);
    s_prefix[tid] = s_and[3] & m0;
    s_mask[tid] = m0;
    s_rem[tid] = static_cast<int>(floor(__dmul_rn(static_cast<double>(n - 1), qs[tid])));
    s_cnt[tid] = n;
    s_open[tid] = n > 1 && fixed_from > 0;
  }
  __syncthreads();
  while (fixed_from > 0) {
    bool open[3];
    bool any = false;
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      open[q] = s_open[q] != 0;
      any |= open[q];
    }
    if (!any) break;
    const int sh = fixed_from > 8 ? fixed_from - 8 : 0;
    const unsigned long long hmask = fixed_from == 64 ? 0ull : (~0ull << fixed_from);
    unsigned long long pre[3], c_or[3], c_and[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      pre[q] = s_prefix[q];
      c_or[q] = 0ull;
      c_and[q] = ~0ull;
    }
    src.visit(tid, [&](unsigned long long k) {
      const unsigned dig = static_cast<unsigned>(k >> sh) & 255u;
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        if (open[q] && (k & hmask) == pre[q]) {
          atomicAdd(&s_hist[q * 256 + dig], 1u);
          c_or[q] |= k;
          c_and[q] &= k;
        }
      }
    });
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      if (open[q]) {
        c_or[q] = warp_or_u64(c_or[q]);
        c_and[q] = warp_and_u64(c_and[q]);
        if (lane == 0) {
          atomicOr(&s_or[q], c_or[q]);
          atomicAnd(&s_and[q], c_and[q]);
        }
      }
    }
    __syncthreads();
    if (warp < 3 && open[warp]) {
      const int q = warp;
      unsigned* hq = s_hist + q * 256 + lane * 8;  // lane owns digits [8 lane, 8 lane + 8)
      unsigned c[8];
      unsigned tot = 0u;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hq[b];
        hq[b] = 0u;  // ready for the next pass
        tot += c[b];
      }
      const unsigned long long cand_or = s_or[q], cand_and = s_and[q];
      const unsigned rem = static_cast<unsigned>(s_rem[q]);
      __syncwarp();
      if (cand_or == cand_and) {  // one distinct key among the candidates
        if (lane == 0) {
          s_prefix[q] = cand_and;
          s_mask[q] = ~0ull;
          s_open[q] = 0;
        }
      } else {
        unsigned incl = tot;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const unsigned v = __shfl_up_sync(0xFFFFFFFFu, incl, o2);
          if (lane >= o2) incl += v;
        }
        unsigned before = incl - tot;
        if (rem >= before && rem < incl) {  // exactly one lane
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            if (rem >= before && rem < before + c[b]) {
              s_prefix[q] |= static_cast<unsigned long long>(lane * 8 + b) << sh;
              s_mask[q] = ~0ull << sh;
              s_rem[q] = static_cast<int>(rem - before);
              s_cnt[q] = static_cast<int>(c[b]);
              s_open[q] = c[b] > 1u && sh > 0;
            }
            before += c[b];
          }
        }
      }
      if (lane == 0) {
        s_or[q] = 0ull;
        s_and[q] = ~0ull;
      }
    }
    fixed_from = sh;
    __syncthreads();
  }
  // Target q's key is its candidates' common value: the one candidate left,
  // or the prefix once all 64 bits are fixed.  The next order statistic is
  // that key again while equal keys remain past the rank, else the smallest
  // key above the candidates' range.
  {
    unsigned long long pre[3], msk[3], lo_min[3], up_min[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      pre[q] = s_prefix[q];
      msk[q] = s_mask[q];
      lo_min[q] = up_min[q] = ~0ull;
    }
    src.visit(tid, [&](unsigned long long k) {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const unsigned long long km = k & msk[q];
        if (km == pre[q]) lo_min[q] = k < lo_min[q] ? k : lo_min[q];
        else if (km > pre[q]) up_min[q] = k < up_min[q] ? k : up_min[q];
      }
    });
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      lo_min[q] = warp_min_u64(lo_min[q]);
      up_min[q] = warp_min_u64(up_min[q]);
    }
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        s_wmin[warp][q] = lo_min[q];
        s_wmin[warp][3 + q] = up_min[q];
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    double r[3];
    for (int qi = 0; qi < 3; ++qi) {
      unsigned long long klo = ~0ull, kup = ~0ull;
      for (int w = 0; w < kDiagWarps; ++w) {
        klo = s_wmin[w][qi] < klo ? s_wmin[w][qi] : klo;
        kup = s_wmin[w][3 + qi] < kup ? s_wmin[w][3 + qi] : kup;
      }
      // each operation rounded on its own, as the formula is written
      const double h = __dmul_rn(static_cast<double>(n - 1), qs[qi]);
      const double fl = floor(h);
      const int lo = static_cast<int>(fl);
      const unsigned long long khi = (lo + 1 < n && s_rem[qi] + 1 >= s_cnt[qi]) ? kup : klo;
      const double xlo = __longlong_as_double(static_cast<long long>(klo));
      const double xhi = __longlong_as_double(static_cast<long long>(khi));
      r[qi] = __dadd_rn(xlo, __dmul_rn(__dsub_rn(h, fl), __dsub_rn(xhi, xlo)));
    }
    o->abs_q50[p] = r[0];
    o->abs_q95[p] = r[1];
    o->abs_q99[p] = r[2];
  }
}

// One launch: blocks [0, 3 S) select the quantiles of (sequence b / 3, pair
// b % 3), the rest compute the per-token sums part by part (the quantile CTAs
// come first so the longest work starts first; the two kinds share no data).
// The kernel is launched programmatically behind the partition kernel: only
// the part CTAs wait for the bases (griddepcontrol.wait).
__global__ void __launch_bounds__(kDiagThreads)
    seg_diag_kernel(const float* __restrict__ A, const float* __restrict__ B,
                    const float* __restrict__ C, const int32_t* __restrict__ tA,
                    const int32_t* __restrict__ tB, const int32_t* __restrict__ tC,
                    const int64_t* __restrict__ offs, const uint8_t* __restrict__ mask, int64_t T,
                    int n_seq, const int* __restrict__ base, double ln_lo, double ln_hi,
                    double cap, double ln_cap, DiagPart* __restrict__ parts,
                    int* __restrict__ cnt_seq, unsigned long long* __restrict__ spill,
                    tim_seq_diag* __restrict__ out, int* status) {
  extern __shared__ unsigned long long keys[];
  const int b = static_cast<int>(blockIdx.x);
  if (b < 3 * n_seq) {
    diag_quantiles(b / 3, b % 3, keys, spill + static_cast<int64_t>(b % 3) * T, A, B, C, offs,
                   mask, T, out);
  } else {
    pdl_wait();  // the partition kernel's bases and zeroed counters
    diag_part(b - 3 * n_seq, keys, A, B, C, tA, tB, tC, offs, mask, T, n_seq, base, ln_lo, ln_hi, cap,
              ln_cap, parts, cnt_seq, out, status);
  }
}

// Diagnostics workspace: status | part bases int32 [S + 1] | per-sequence part
// counters int32 [S] (zeroed by the partition kernel of each call) | parts |
// quantile keys past the shared-memory ones, uint64 [3][T] (pair p, token t).
size_t diag_base_offset() { return 1024; }
size_t diag_counter_offset(int n_seq) {
  return align_up(diag_base_offset() + static_cast<size_t>(n_seq + 1) * 4, 256);
}
size_t diag_parts_offset(int n_seq) {
  return align_up(diag_counter_offset(n_seq) + static_cast<size_t>(n_seq) * 4, 1024);
}
size_t diag_spill_offset(int64_t T, int n_seq) {
  return align_up(diag_parts_offset(n_seq) +
                      static_cast<size_t>(seq_parts_bound(T, n_seq)) * sizeof(DiagPart),
                  1024);
}
size_t diag_workspace_bytes(int64_t T, int n_seq) {
  return align_up(diag_spill_offset(T, n_seq) + 3 * static_cast<size_t>(T) * 8, 1024);
}

cudaError_t launch_seg_diag(const float* A, const float* B, const float* C, const int32_t* tA,
                            const int32_t* tB, const int32_t* tC, const int64_t* offs, int n_seq,
                            const uint8_t* mask, int64_t T, float tis_cap, float mis_lo,
                            float mis_hi, tim_seq_diag* out, void* workspace,
                            cudaStream_t stream) {
  const double cap = static_cast<double>(tis_cap);
  int* status = static_cast<int*>(workspace);
  int* base = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + diag_base_offset());
  DiagPart* parts =
      reinterpret_cast<DiagPart*>(static_cast<uint8_t*>(workspace) + diag_parts_offset(n_seq));
  int* cnt_seq =
      reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + diag_counter_offset(n_seq));
  unsigned long long* spill = reinterpret_cast<unsigned long long*>(
      static_cast<uint8_t*>(workspace) + diag_spill_offset(T, n_seq));
  cudaError_t err = launch_seq_partition(offs, n_seq, T, base, cnt_seq, stream);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(seg_diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kDiagSmemBytes));
  if (err != cudaSuccess) return err;
  const int64_t blocks = 3 * static_cast<int64_t>(n_seq) + seq_parts_bound(T, n_seq);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kDiagThreads);
  cfg.dynamicSmemBytes = kDiagSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, seg_diag_kernel, A, B, C, tA, tB, tC, offs, mask, T, n_seq,
                            static_cast<const int*>(base), std::log(static_cast<double>(mis_lo)),
                            std::log(static_cast<double>(mis_hi)), cap, std::log(cap), parts,
                            cnt_seq, spill, out, status);
}

}  // namespace tim
