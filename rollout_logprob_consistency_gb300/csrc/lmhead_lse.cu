// Stage 2 of the linear logprob: LM-head GEMM z = y . W^T on the tcgen05 tensor
// cores, with a fused epilogue that reduces every 256-column vocabulary tile of
// every row to softmax statistics, so the [T, V] logits never reach memory.
//
// Sources: "Debugging Logprob Mismatches in LLM Reinforcement Learning", Case 2
// (selected-token logprob = chosen logit minus the log of the summed
// exponentials over the whole vocabulary) and "How this differs from a real
// temperature mismatch" (temperature scales the logits before the softmax);
// "Training and rollout stop disagreeing: vime and RL-Kernel ...",
// Interpretation (GEMM K-dimension reduction and accumulation precision fixed;
// linear logprob over the true vocabulary range); "Rollout-Training Mismatch in
// LLM RL", section 5.2 (no small-batch backend switch; batch-invariant
// accumulation).
//
// Design (one CTA per SM, persistent over (row-tile, vocab-tile) work items):
//   warp 0       TMA producer: y tile [128 x 64] and W tile [256 x 64] per
//                stage, 128-byte swizzle, 4-stage mbarrier ring.
//   warp 1       allocates 512 TMEM columns; one thread issues
//                tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16; bf16
//                in, fp32 accumulate) 4x per stage into one of two 256-column
//                accumulators, then tcgen05.commit.
//   warps 2..5   epilogue, one thread per TMEM lane = one row: reads 32 columns
//                at a time (tcgen05.ld 32x32b.x32), keeps an online max / sum of
//                2^(z*log2e/tau - max), the arg-max of the raw logits and the
//                target's logit, and writes one 16-byte record per (row, tile).
//   Double-buffered accumulators let the epilogue of tile i overlap the MMAs of
//   tile i+1.
//   Row-tile pairs (two 128-row tiles against one W tile, see kPrecBf16x2) use
//   both accumulators for one work item and eight epilogue warps: warps 2..5
//   read the first row tile's accumulator, warps 6..9 the second's.
//
// Batch invariance: every logit is the same sequence of MMAs (k-blocks in
// order, 4 K=16 steps each) whatever T is; rows past T (zeros written by the
// RMSNorm kernel up to the next 128-row boundary) never touch other rows; the
// epilogue arithmetic of a (row, tile) pair is fixed.  Which CTA computes a
// tile does not matter.
//
// The same kernel serves the other paths through two template parameters:
//   kMode  0 scoring records (above); 1 candidate collection and 4 top-4
//          records (processed score); 2 logit gradient and 3 plain fp32-output
//          GEMM (backward);
//   kPrec  bf16 (above), e4m3 codes with power-of-two row scales (FP8 head),
//          or fp32 operands as three tf32 products (FP32 head).
// Only the operand staging, the MMA kind and the epilogue differ; the tile
// shape, the ring, the accumulator hand-off and the raster are shared.
//
// Launched with programmatic stream serialisation when the batch fits one
// raster group: the producer streams its first W stages, then waits
// (griddepcontrol.wait, a no-op for an ordinary launch) for the RMSNorm kernel
// before the first load of y.
//
// Every mbarrier wait is bounded (2 s by default); on timeout the kernel
// records TIM_ERR_TIMEOUT, raises a CTA-wide abort flag, waits (bounded) for
// its own TMA copies and MMAs still in flight, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>

#include "tim_common.cuh"

namespace tim {

struct GemmArgs {
  int64_t T;
  int v0;     // global vocabulary id of W row 0 (0 unless W is a vocabulary shard)
  int v_end;  // global end (exclusive) of the vocabulary columns this launch scores
  int d;
  int num_m;
  int num_n;
  int num_kb;
  int group_m;
  int64_t num_tiles;
  float k2;        // log2(e) / temperature
  float inv_temp;  // 1 / temperature
  const int32_t* ids;
  float4* part;
  float* tgt;
  int* status;
  // collect mode only: per-row logit threshold, candidate counters, candidate
  // slots (logit bits, vocabulary id) [T][cap]
  const float* thr;
  int* cnt;
  uint2* cand;
  int cap;
  // e4m3 operands only: per-row scales of y and per-vocabulary-row scales of W
  const float* sy;
  const float* sw;
  // logit-gradient mode only: forward lse [T] and upstream gradient [T]; output
  // G = dL/dz in bf16, row-major [rows_padded(T)][ldg]
  const float* lse;
  const float* gup;
  uint16_t* gz;
  int64_t ldg;
  // store mode only: C fp32 [T][ldc] (T = rows of A, v_end = columns), C = A.B^T
  // or C += A.B^T; a_mn / b_mn: that operand is stored MN-major ([K][rows],
  // rows contiguous) instead of K-major
  float* c;
  int64_t ldc;
  int accumulate;
  int a_mn;
  int b_mn;
  // bounded-wait limit of every mbarrier wait; the wait self-test shortens it and
  // sets stall_producer so that no load is ever issued
  uint64_t wait_limit_ns;
  int stall_producer;
  // scoring-type launches within one raster group: the CTA that works on a W
  // tile's first work item prefetches that tile's W k-blocks into L2 this many
  // k-blocks ahead of its loads (0 = none); the other CTAs on the tile then find
  // them in L2
  int w_prefetch;
  // top-4 mode only: per-(row, tile) records of the four largest logits
  void* top4;
  // collect mode only: when dyn_T is set, only row tiles below *dyn_T (a row
  // count written by an earlier kernel) are computed, and local row r stands for
  // row row_map[r] of the candidate slots and thresholds
  const int* dyn_T;
  const int* row_map;
};


// Operand precision of the GEMM.
//   kPrecBf16   bf16 y and W, kind::f16, 64 K-elements per 128-byte stage row.
//   kPrecE4m3   e4m3 codes, kind::f8f6f4, 128 K-elements per stage row; the
//               epilogue multiplies each logit by s_y[row] * s_W[col] (powers of
//               two, so the scaling is exact).
//   kPrecTf32x3 fp32 y and W, each given as a tf32 part (low 13 mantissa bits
//               cleared) and the exact fp32 remainder; kind::tf32 computes
//               big*big + big*small + small*big per K step, 32 K-elements per
//               stage row; a stage holds both parts of both operands, so the
//               ring has half as many stages in the same shared memory.
//   kPrecBf16x2 bf16 as kPrecBf16, but a work item is a pair of row tiles
//               (2m, 2m + 1) against one W tile: a stage holds both y tiles and
//               one W tile (64 KiB, 3 stages), and every K step issues the same
//               M=128 MMA once per row tile into its own accumulator.  Each row
//               sees the identical MMA sequence of the one-tile form; only the
//               number of CTAs that stream a W tile at once changes (the scoring
//               mode, see plan_scoring_schedule, and the backward products).
enum Prec : int { kPrecBf16 = 0, kPrecE4m3 = 1, kPrecTf32x3 = 2, kPrecBf16x2 = 3 };

template <int kPrec>
struct StageGeom {
  static constexpr int kParts = kPrec == kPrecTf32x3 ? 2 : 1;
  static constexpr int kRowTiles = kPrec == kPrecBf16x2 ? 2 : 1;  // row tiles per work item
  static constexpr int kStageA = kParts * kRowTiles * kABytes;
  static constexpr int kStageB = kParts * kBBytes;
  static constexpr int kS = kStages * (kABytes + kBBytes) / (kStageA + kStageB);
  static constexpr int kKElems = kPrec == kPrecE4m3 ? 2 * kBK : kPrec == kPrecTf32x3 ? kBK / 2 : kBK;
  // epilogue warps: one per TMEM lane quadrant and accumulator (a pair's two
  // accumulators are read side by side by two warp groups)
  static constexpr int kEpi = kRowTiles * kEpiWarps;
  static constexpr int kThreads = 64 + 32 * kEpi;
  // TMEM per tile: one 256-column fp32 accumulator, double-buffered; the tf32x3
  // path adds a second 256-column accumulator for the two correction products
  // (big*small + small*big), so its tile takes all 512 columns, single-buffered.
  // Keeping the corrections apart leaves the main sum with d/8 accumulation
  // steps instead of 3d/8 (each step of the tensor-core accumulation costs up to
  // one rounding of the running sum).
  // The row-tile pair likewise takes all 512 columns: one accumulator per row tile.
  static constexpr int kAccCols = (kPrec == kPrecTf32x3 || kPrec == kPrecBf16x2) ? 2 * kBN : kBN;
  static constexpr int kNumAcc = kTmemCols / kAccCols;
};
static_assert(StageGeom<kPrecBf16>::kS == kStages && StageGeom<kPrecTf32x3>::kS == 2 &&
                  StageGeom<kPrecBf16x2>::kS == 3,
              "stage rings fill the same shared memory");

constexpr size_t kGemmSmemBytes =
    1024 /* alignment slack */ + kStages * (kABytes + kBBytes) + 256 /* barriers, flags */;
// The logit-gradient mode also stages each epilogue warp's 32 x 32 bf16 block of G
// (2 KB per warp) so that its row-major stores cover whole 32-byte sectors.
constexpr size_t kGradStageBytes = kEpiWarps * 32 * 64;

__host__ __device__ constexpr size_t gemm_smem_bytes(int mode) {
  return kGemmSmemBytes + (mode == 2 ? kGradStageBytes : 0);
}

// MN-major operand tile (store mode): boxes of 64 rows of K x 64 bf16 of M or N
// (128-byte rows, 128-byte swizzle), one box per 64 elements of M or N.
constexpr int kMnChunkBytes = 64 * 128;

// Shared-memory descriptor of an MN-major 128-byte-swizzled bf16 tile: within
// an 8-row atom (1024 bytes) each row holds 64 consecutive elements of M or N
// for one k; the leading-dimension offset steps to the next 64 elements of M or
// N (the next box, kMnChunkBytes), the stride-dimension offset to the next 8
// rows of K (1024 bytes).  Checked bit for bit against a CPU product on
// small-integer tiles for A, B and both MN-major.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  desc |= static_cast<uint64_t>(kMnChunkBytes >> 4) << 16;
  desc |= static_cast<uint64_t>(1024u >> 4) << 32;
  desc |= static_cast<uint64_t>(1u) << 46;
  desc |= static_cast<uint64_t>(2u) << 61;
  return desc;
}

__device__ __forceinline__ void tile_coords(int64_t tile, const GemmArgs& a, int& m, int& n) {
  const int64_t per_group = static_cast<int64_t>(a.group_m) * a.num_n;
  const int64_t g = tile / per_group;
  const int64_t r = tile - g * per_group;
  const int m0 = static_cast<int>(g * a.group_m);
  const int gm = min(a.group_m, a.num_m - m0);
  m = m0 + static_cast<int>(r % gm);
  n = static_cast<int>(r / gm);
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* status) {
  set_status(status, TIM_ERR_TIMEOUT);
  *abort_flag = 1;
  __threadfence_block();
}

// Bounded wait that ignores the abort flag (used while winding down).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// One 32-column chunk of one row: update the running (max, sum) in the base-2
// domain, the arg-max of the raw logits (first occurrence), and pick the
// target's logit if it lies in this chunk.
template <bool kPartial>
__device__ __forceinline__ void epilogue_chunk(const uint32_t (&r)[32], int nvalid, int col0,
                                               int rel_c, float k2, float& m2, float& sum,
                                               float& bz, int& bi, float& zt) {
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    v[j] = __uint_as_float(r[j]);
    if (kPartial) v[j] = (j < nvalid) ? v[j] : -INFINITY;
  }
  // chunk maximum; its first index is looked up only when it beats the row's best
  // so far (the arg-max is then the first index of the largest logit, as a
  // sequential scan gives; outputs bitwise equal to the scan with an index per
  // logit, which took three instructions a logit instead of one)
  float cmax = v[0];
#pragma unroll
  for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, v[j]);
  const float mnew = fmaxf(m2, cmax * k2);
  float cs = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) cs += ex2_approx(fmaf(v[j], k2, -mnew));
  sum = sum * ex2_approx(m2 - mnew) + cs;
  m2 = mnew;
  if (cmax > bz) {
    int cidx = 31;
#pragma unroll
    for (int j = 30; j >= 0; --j)
      if (v[j] == cmax) cidx = j;
    bz = cmax;
    bi = col0 + cidx;
  }
  if (static_cast<unsigned>(rel_c) < 32u) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j == rel_c) zt = v[j];
  }
}

// kMode 0: per-(row, tile) softmax records and the target logit (the scoring path).
// kMode 1: candidate collection -- every logit >= the row's threshold is appended
//          (in no particular order) to the row's candidate slots; used by the
//          processed (top-k / top-p) score, which sorts the candidates afterwards.
// kMode 2: logit gradient of the backward -- G = (g_t / tau)(1[v = x_t] - p_tv)
//          with p = exp(z / tau - lse_t), written once in bf16, row-major
//          (rows T .. rows_padded(T)-1 get zeros).
// kMode 3: plain GEMM C (+)= A . B^T stored in fp32 (the two backward products).
// kMode 4: top-4 records -- the four largest logits of every (row, tile) and
//          their ids (the first pass of the processed score).
// kPrec: operand precision (see Prec).  tmap_y2 / tmap_w2 are the remainder
// parts for kPrecTf32x3 and unused otherwise.
template <int kMode, int kPrec>
__global__ void __launch_bounds__(StageGeom<kPrec>::kThreads, 1)
    lmhead_lse_kernel(const __grid_constant__ CUtensorMap tmap_y,
                      const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_y2,
                      const __grid_constant__ CUtensorMap tmap_w2, const GemmArgs a) {
  using G = StageGeom<kPrec>;
  constexpr bool kFp8 = kPrec == kPrecE4m3;
  constexpr bool kX3 = kPrec == kPrecTf32x3;
  constexpr int kRT = G::kRowTiles;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + G::kS * G::kStageA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + G::kS * G::kStageB);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  uint32_t* last_parity = reinterpret_cast<uint32_t*>(tmem_holder + 2);  // [kStages], producer
  uint8_t* grad_stage = reinterpret_cast<uint8_t*>(bars) + 256;  // mode 2 only

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int kKElems = G::kKElems;  // K elements per 128-byte stage row
  constexpr uint32_t kTx = G::kStageA + G::kStageB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::kS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      last_parity[s] = 0xFFFFFFFFu;  // no load issued into this stage yet
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], G::kEpi);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    prefetch_tmap(&tmap_y);
    prefetch_tmap(&tmap_w);
    if (kX3) {
      prefetch_tmap(&tmap_y2);
      prefetch_tmap(&tmap_w2);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // rows actually present (collect mode with a device-side row count)
  const int64_t t_rows = (kMode == 1 && a.dyn_T != nullptr) ? static_cast<int64_t>(*a.dyn_T) : a.T;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !a.stall_producer) {
      // One stage of each operand: a K-major tile is one box (128-byte rows of K,
      // 8-row swizzle atoms); an MN-major tile (store mode) is boxes of 64 rows of
      // K x 64 elements of M or N, placed kMnChunkBytes apart.
      // mt: first row tile of the work item; two: the item's second row tile
      // exists (row-tile pairs only)
      auto load_a = [&](int st, int kb, int mt, bool two) {
        uint8_t* dst = sA + st * G::kStageA;
        if constexpr (kMode == 3) {
          if (a.a_mn) {
#pragma unroll
            for (int h = 0; h < kRT; ++h) {
              if (h > 0 && !two) break;
#pragma unroll
              for (int c = 0; c < kBM / 64; ++c)
                tma_load_2d(dst + h * kABytes + c * kMnChunkBytes, &tmap_y,
                            (mt + h) * kBM + c * 64, kb * kKElems, &full[st]);
            }
            return;
          }
        }
        tma_load_2d(dst, &tmap_y, kb * kKElems, mt * kBM, &full[st]);
        if (kX3) tma_load_2d(dst + kABytes, &tmap_y2, kb * kKElems, mt * kBM, &full[st]);
        if (kRT == 2 && two)
          tma_load_2d(dst + kABytes, &tmap_y, kb * kKElems, (mt + 1) * kBM, &full[st]);
      };
      auto load_b = [&](int st, int kb, int n) {
        uint8_t* dst = sB + st * G::kStageB;
        if constexpr (kMode == 3) {
          if (a.b_mn) {
#pragma unroll
            for (int c = 0; c < kBN / 64; ++c)
              tma_load_2d(dst + c * kMnChunkBytes, &tmap_w, n * kBN + c * 64, kb * kKElems,
                          &full[st]);
            return;
          }
        }
        tma_load_2d(dst, &tmap_w, kb * kKElems, n * kBN, &full[st]);
        if (kX3) tma_load_2d(dst + kBBytes, &tmap_w2, kb * kKElems, n * kBN, &full[st]);
      };
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      bool first = true;
      for (int64_t tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x) {
        int m, n;
        tile_coords(tile, a, m, n);
        const int mt = m * kRT;
        if (static_cast<int64_t>(mt) * kBM >= t_rows) continue;  // no rows in this tile
        const bool two = kRT == 2 && static_cast<int64_t>(mt + 1) * kBM < t_rows;
        const uint32_t tx = (kRT == 1 || two) ? kTx : kTx - kABytes;
        int kb0 = 0;
        if (first) {
          // W does not depend on the RMSNorm kernel that precedes this one in the
          // stream: stream the first stages of W before waiting for y to be ready.
          const int pre = min(G::kS, a.num_kb);
          for (int s = 0; s < pre; ++s) {
            mbar_arrive_expect_tx(&full[s], tx);
            load_b(s, s, n);
          }
          pdl_wait();
          for (int s = 0; s < pre; ++s) {
            load_a(s, s, mt, two);
            last_parity[s] = 0;
          }
          stage = pre % G::kS;
          ph = (pre == G::kS) ? 1u : 0u;
          kb0 = pre;
          first = false;
        }
        // the CTA on the W tile's first work item of the raster group prefetches
        const bool leader = a.w_prefetch > 0 && (m % a.group_m) == 0;
        if (leader) {
          for (int k = kb0 + 1; k < min(a.num_kb, kb0 + a.w_prefetch); ++k)
            tma_prefetch_2d(&tmap_w, k * kKElems, n * kBN);
        }
        for (int kb = kb0; kb < a.num_kb; ++kb) {
          if (leader && kb + a.w_prefetch < a.num_kb)
            tma_prefetch_2d(&tmap_w, (kb + a.w_prefetch) * kKElems, n * kBN);
          if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], tx);
          load_a(stage, kb, mt, two);
          load_b(stage, kb, n);
          last_parity[stage] = ph;
          if (++stage == G::kS) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) raise_abort(abort_flag, a.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t idesc = kFp8  ? umma_idesc_e4m3_f32(kBM, kBN)
                       : kX3 ? umma_idesc_tf32_f32(kBM, kBN)
                             : umma_idesc_bf16_f32(kBM, kBN);
      if constexpr (kMode == 3)  // bits 15 / 16: A / B major (1 = MN)
        idesc |= (a.a_mn ? (1u << 15) : 0u) | (a.b_mn ? (1u << 16) : 0u);
      int stage = 0;
      uint32_t ph = 0;
      uint32_t acc = 0, acc_ph = 0;
      bool ok = true;
      for (int64_t tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x) {
        if (kMode == 1 && a.dyn_T != nullptr) {
          int m, n;
          tile_coords(tile, a, m, n);
          if (static_cast<int64_t>(m) * kBM >= t_rows) continue;
        }
        bool two = false;  // row-tile pairs: the item's second row tile exists
        if constexpr (kRT == 2) {
          int m, n;
          tile_coords(tile, a, m, n);
          two = static_cast<int64_t>(2 * m + 1) * kBM < t_rows;
        }
        if (!mbar_wait(&acc_empty[acc], acc_ph ^ 1u, abort_flag, a.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * G::kAccCols;
        for (int kb = 0; kb < a.num_kb; ++kb) {
          if (!mbar_wait(&full[stage], ph, abort_flag, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * G::kStageA);
          const uint32_t b0 = smem_u32(sB + stage * G::kStageB);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 4 x 32 bytes of K per 128-byte row
            const uint32_t acc_k = (kb | k) != 0 ? 1u : 0u;
            if constexpr (kFp8) {
              umma_e4m3(d_tmem, sw128_kmajor_desc(a0 + k * 32), sw128_kmajor_desc(b0 + k * 32),
                        idesc, acc_k);
            } else if constexpr (kX3) {
              const uint64_t ab = sw128_kmajor_desc(a0 + k * 32);
              const uint64_t as = sw128_kmajor_desc(a0 + kABytes + k * 32);
              const uint64_t bb = sw128_kmajor_desc(b0 + k * 32);
              const uint64_t bs = sw128_kmajor_desc(b0 + kBBytes + k * 32);
              umma_tf32(d_tmem, ab, bb, idesc, acc_k);
              umma_tf32(d_tmem + kBN, ab, bs, idesc, acc_k);
              umma_tf32(d_tmem + kBN, as, bb, idesc, 1u);
            } else {
              uint64_t ad = sw128_kmajor_desc(a0 + k * 32);
              uint64_t bd = sw128_kmajor_desc(b0 + k * 32);
              uint64_t ad2 = sw128_kmajor_desc(a0 + kABytes + k * 32);  // row-tile pairs
              if constexpr (kMode == 3) {  // 16 K-rows of an MN-major tile: 2 atoms
                if (a.a_mn) {
                  ad = sw128_mnmajor_desc(a0 + k * 2048);
                  ad2 = sw128_mnmajor_desc(a0 + kABytes + k * 2048);
                }
                if (a.b_mn) bd = sw128_mnmajor_desc(b0 + k * 2048);
              }
              umma_bf16(d_tmem, ad, bd, idesc, acc_k);
              if (kRT == 2 && two)  // same B slice, second row tile, own accumulator
                umma_bf16(d_tmem + kBN, ad2, bd, idesc, acc_k);
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == G::kS) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);
        if (++acc == static_cast<uint32_t>(G::kNumAcc)) {
          acc = 0;
          acc_ph ^= 1u;
        }
      }
      if (!ok) raise_abort(abort_flag, a.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    // row tile of the work item this warp reads: 0, or with row-tile pairs 0 for
    // warps 2-5 and 1 for warps 6-9 (one accumulator each, kBN columns apart)
    const int h = (warp - 2) / kEpiWarps;
    uint32_t acc = 0, acc_ph = 0;
    for (int64_t tile = blockIdx.x; tile < a.num_tiles; tile += gridDim.x) {
      int m, n;
      tile_coords(tile, a, m, n);
      const int mt = m * kRT;  // first row tile of the work item
      if (static_cast<int64_t>(mt) * kBM >= t_rows) continue;
      // a pair's second row tile may not exist: its warps then only take part in
      // the accumulator hand-off
      const int nchunk = static_cast<int64_t>(mt + h) * kBM < t_rows ? kBN / 32 : 0;
      const int64_t row = static_cast<int64_t>(mt + h) * kBM + q * 32 + lane;
      const int x = (kMode != 3 && row < a.T) ? __ldg(a.ids + row) : -1;
      const int col_base = a.v0 + n * kBN;  // global vocabulary id of the tile's column 0
      const int rel = x - col_base;

      int ok = 1;
      if (lane == 0) ok = mbar_wait(&acc_full[acc], acc_ph, abort_flag, a.wait_limit_ns) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) raise_abort(abort_flag, a.status);
        break;
      }
      tc_fence_after();
      __syncwarp();

      float m2 = -INFINITY, sum = 0.f, bz = -INFINITY, zt = 0.f;
      int bi = col_base;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             acc * G::kAccCols + h * kBN;
      if constexpr (kMode == 0 && !kFp8 && !kX3) {
        // bf16 operands: the load of chunk c + 1 is in flight while chunk c is
        // reduced (same chunks, same order, same arithmetic as one load at a time)
        const int nch = min(nchunk, max(0, (a.v_end - col_base + 31) / 32));
        auto reduce = [&](const uint32_t(&r)[32], int c) {
          const int col0 = col_base + c * 32;
          const int nvalid = min(32, a.v_end - col0);
          if (nvalid == 32)
            epilogue_chunk<false>(r, 32, col0, rel - c * 32, a.k2, m2, sum, bz, bi, zt);
          else
            epilogue_chunk<true>(r, nvalid, col0, rel - c * 32, a.k2, m2, sum, bz, bi, zt);
        };
        uint32_t ra[32], rb[32];
        if (nch > 0) {
          tmem_ld32_async(tbase, ra);
          tmem_ld_wait(ra);
        }
#pragma unroll 1
        for (int c = 0; c < nch; c += 2) {
          if (c + 1 < nch) tmem_ld32_async(tbase + (c + 1) * 32, rb);
          reduce(ra, c);
          if (c + 1 < nch) {
            tmem_ld_wait(rb);
            if (c + 2 < nch) tmem_ld32_async(tbase + (c + 2) * 32, ra);
            reduce(rb, c + 1);
            if (c + 2 < nch) tmem_ld_wait(ra);
          }
        }
      } else if constexpr (kMode == 0) {
        const float srow = kFp8 ? __ldg(a.sy + row) : 1.f;
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          const int col0 = col_base + c * 32;
          if (col0 >= a.v_end) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          const int nvalid = min(32, a.v_end - col0);
          if constexpr (kFp8) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float sc = srow * __ldg(a.sw + min(col0 + j, a.v_end - 1));
              r[j] = __float_as_uint(__uint_as_float(r[j]) * sc);
            }
          }
          if constexpr (kX3) {
            uint32_t rc[32];
            tmem_ld32(tbase + kBN + c * 32, rc);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              r[j] = __float_as_uint(__uint_as_float(r[j]) + __uint_as_float(rc[j]));
          }
          if (nvalid == 32)
            epilogue_chunk<false>(r, 32, col0, rel - c * 32, a.k2, m2, sum, bz, bi, zt);
          else
            epilogue_chunk<true>(r, nvalid, col0, rel - c * 32, a.k2, m2, sum, bz, bi, zt);
        }
      } else if constexpr (kMode == 2) {
        const bool live = row < a.T;
        const bool bad = live && (x < 0 || x >= a.v_end);
        if (bad) set_status(a.status, TIM_ERR_TOKEN_RANGE);
        const float gs = (live && !bad) ? __ldg(a.gup + row) * a.inv_temp : 0.f;
        const float l2 = live ? __ldg(a.lse + row) * 1.4426950408889634f : 0.f;
        const uint64_t pol = l2_policy_evict_first();
        // this warp's staging block: row l (= lane) holds 4 x 16 bytes, stored at
        // 16-byte slot (w ^ ((l >> 1) & 3)) -- conflict-free writes by row and
        // reads by (row, quarter)
        uint8_t* stg = grad_stage + q * (32 * 64);
        const int64_t row0 = row - lane;  // first row of this warp's 32
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          const int col0 = col_base + c * 32;
          if (col0 >= a.v_end) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          const int nvalid = min(32, a.v_end - col0);
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float gv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const float p = ex2_approx(fmaf(__uint_as_float(r[j + u]), a.k2, -l2));
              const float oh = (col0 + j + u == x) ? 1.f : 0.f;
              gv[u] = (j + u < nvalid) ? gs * (oh - p) : 0.f;
            }
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(gv[0]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(gv[1]));
            packed[j >> 1] = lo | (hi << 16);
          }
#pragma unroll
          for (int w = 0; w < 4; ++w)
            *reinterpret_cast<uint4*>(stg + lane * 64 + ((w ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2],
                           packed[4 * w + 3]);
          __syncwarp();
          // 4 stores, each writing 8 rows x 64 bytes (whole sectors)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = 8 * i + (lane >> 2), qq = lane & 3;
            const uint4 v =
                *reinterpret_cast<const uint4*>(stg + r * 64 + ((qq ^ ((r >> 1) & 3)) << 4));
            st_global_v4_hint(a.gz + (row0 + r) * a.ldg + col0 + qq * 8, v, pol);
          }
          __syncwarp();
        }
      } else if constexpr (kMode == 3) {
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          const int col0 = col_base + c * 32;
          if (col0 >= a.v_end) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          if (row < a.T) {
            float4* dst = reinterpret_cast<float4*>(a.c + row * a.ldc + col0);
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              float4 v = make_float4(__uint_as_float(r[4 * w]), __uint_as_float(r[4 * w + 1]),
                                     __uint_as_float(r[4 * w + 2]), __uint_as_float(r[4 * w + 3]));
              if (a.accumulate) {
                const float4 o = dst[w];
                v.x += o.x;
                v.y += o.y;
                v.z += o.z;
                v.w += o.w;
              }
              dst[w] = v;
            }
          }
        }
      } else if constexpr (kMode == 4) {
        float tv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        int ti[4] = {-1, -1, -1, -1};
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          const int col0 = col_base + c * 32;
          if (col0 >= a.v_end) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          const int nvalid = min(32, a.v_end - col0);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float cv = j < nvalid ? __uint_as_float(r[j]) : -INFINITY;
            if (cv > tv[3]) {  // insert; strict > keeps the earlier (lower) id first on ties
              int ci = col0 + j;
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                if (cv > tv[p]) {
                  const float fv = tv[p];
                  const int fi = ti[p];
                  tv[p] = cv;
                  ti[p] = ci;
                  cv = fv;
                  ci = fi;
                }
              }
            }
          }
        }
        if (row < a.T) {
          Top4Rec* rec = static_cast<Top4Rec*>(a.top4) + ((row >> 5) * a.num_n + n) * 32 + (row & 31);
          *reinterpret_cast<float4*>(rec->v) = make_float4(tv[0], tv[1], tv[2], tv[3]);
          *reinterpret_cast<int4*>(rec->id) = make_int4(ti[0], ti[1], ti[2], ti[3]);
        }
      } else {
        const bool live = row < t_rows;
        const int64_t orow = (live && a.row_map != nullptr) ? __ldg(a.row_map + row) : row;
        const float thr = live ? __ldcg(a.thr + orow) : INFINITY;
#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
          const int col0 = col_base + c * 32;
          if (col0 >= a.v_end) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          const int nvalid = min(32, a.v_end - col0);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < nvalid && live && __uint_as_float(r[j]) >= thr) {
              const int slot = atomicAdd(a.cnt + orow, 1);
              if (slot < a.cap) a.cand[orow * a.cap + slot] = make_uint2(r[j], col0 + j);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);

      if (kMode == 0 && row < a.T) {
        a.part[((row >> 5) * a.num_n + n) * 32 + (row & 31)] =
            make_float4(m2, sum, bz, __int_as_float(bi));
        if (static_cast<unsigned>(rel) < static_cast<unsigned>(kBN)) a.tgt[row] = zt * a.inv_temp;
      }
      if (++acc == static_cast<uint32_t>(G::kNumAcc)) {
        acc = 0;
        acc_ph ^= 1u;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && lane == 0) {
      // wait for TMA copies still landing in shared memory
      for (int s = 0; s < G::kS; ++s)
        if (last_parity[s] != 0xFFFFFFFFu) mbar_wait_drain(&full[s], last_parity[s]);
    }
    if (warp == 1 && lane == 0) {
      // wait for MMAs still reading shared memory / writing TMEM
      umma_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side

// The driver's tensor-map encoder, resolved on first use and cached; host threads
// may call concurrently (the cache is atomic, and a failed lookup is retried).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cache{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cache.load(std::memory_order_acquire);
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      cache.store(fn, std::memory_order_release);
    }
  }
  return fn;
}

// [rows, d] row-major operand (bf16; e4m3 codes; fp32 for the tf32 parts), box =
// one 128-byte row of K x box_rows rows with 128-byte swizzle; rows past the end
// read as zeros.
static bool make_kmajor_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t d,
                            uint32_t box_rows, int prec) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const uint64_t esize = prec == kPrecE4m3 ? 1 : prec == kPrecTf32x3 ? 4 : 2;
  const CUtensorMapDataType dt = prec == kPrecE4m3     ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : prec == kPrecTf32x3 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t dims[2] = {d, rows};
  const cuuint64_t strides[1] = {d * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 [rows, K] operand with row stride ld elements (ld * 2 a multiple of 16);
// columns K .. and rows past `rows` read as zeros.
static bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K,
                          uint64_t ld, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 operand stored MN-major: [K][ld] with its mn_extent rows of the product
// (M or N) contiguous; box = 64 elements of M or N x 64 rows of K, 128-byte
// swizzle; elements past mn_extent or rows past k_extent read as zeros.
static bool make_bf16_mn_map(CUtensorMap* map, const void* base, uint64_t mn_extent,
                             uint64_t k_extent, uint64_t ld) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {mn_extent, k_extent};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int kMode, int kPrec>
static cudaError_t launch_gemm(const CUtensorMap& map_y, const CUtensorMap& map_w,
                               const CUtensorMap& map_y2, const CUtensorMap& map_w2,
                               const GemmArgs& a, cudaStream_t stream, int num_sms,
                               bool programmatic) {
  cudaError_t e = cudaFuncSetAttribute(lmhead_lse_kernel<kMode, kPrec>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(gemm_smem_bytes(kMode)));
  if (e != cudaSuccess) return e;
  const int64_t grid = a.num_tiles < num_sms ? a.num_tiles : num_sms;
  // Programmatic dependent launch: the kernel's prologue and its first W loads
  // may overlap the tail of the RMSNorm kernel; y is read only after
  // griddepcontrol.wait.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(StageGeom<kPrec>::kThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(kMode);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, lmhead_lse_kernel<kMode, kPrec>, map_y, map_w, map_y2, map_w2,
                            a);
}

static cudaError_t make_args(GemmArgs& a, CUtensorMap& map_y, CUtensorMap& map_w, const void* y,
                             const void* W, const int32_t* ids, int64_t T, int d, int V, int v0,
                             float temperature, int* status, int prec = kPrecBf16) {
  if (!make_kmajor_map(&map_y, y, static_cast<uint64_t>(rows_padded(T)),
                       static_cast<uint64_t>(d), kBM, prec) ||
      !make_kmajor_map(&map_w, W, static_cast<uint64_t>(V), static_cast<uint64_t>(d), kBN, prec))
    return cudaErrorInvalidValue;
  a.T = T;
  a.v0 = v0;
  a.v_end = v0 + V;
  a.d = d;
  a.num_m = static_cast<int>((T + kBM - 1) / kBM);
  a.num_n = (V + kBN - 1) / kBN;
  a.num_kb = prec == kPrecE4m3     ? d / StageGeom<kPrecE4m3>::kKElems
             : prec == kPrecTf32x3 ? d / StageGeom<kPrecTf32x3>::kKElems
                                   : d / StageGeom<kPrecBf16>::kKElems;
  // Raster groups of row tiles that sweep the vocabulary together (each group
  // streams W once and keeps its y tiles in L2).  Measured on GB300: 48 row tiles
  // at d <= 4096 (d = 4096: 36-48 equal, 64 10% slower); 36 at larger d (d = 5120:
  // 116-118 ms per 131072 rows with 28-36, 130 ms with 48).  The fp32 operands of
  // the tf32x3 path are four times the bytes of bf16 ones, so their group is a
  // quarter (d = 4096: 136 ms with 12 row tiles, 145 ms with 48, 168 ms with 96);
  // e4m3 operands do as well with 48 as with 96.
  a.group_m = d <= 4096 ? 48 : 36;
  if (prec == kPrecTf32x3) a.group_m /= 4;
  a.w_prefetch = 0;
  a.num_tiles = static_cast<int64_t>(a.num_m) * a.num_n;
  a.k2 = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  a.inv_temp = static_cast<float>(1.0 / static_cast<double>(temperature));
  a.ids = ids;
  a.part = nullptr;
  a.tgt = nullptr;
  a.status = status;
  a.thr = nullptr;
  a.cnt = nullptr;
  a.cand = nullptr;
  a.cap = 0;
  a.sy = nullptr;
  a.sw = nullptr;
  a.lse = nullptr;
  a.gup = nullptr;
  a.gz = nullptr;
  a.ldg = 0;
  a.c = nullptr;
  a.ldc = 0;
  a.accumulate = 0;
  a.a_mn = 0;
  a.b_mn = 0;
  a.wait_limit_ns = kWaitLimitNs;
  a.stall_producer = 0;
  a.top4 = nullptr;
  a.dyn_T = nullptr;
  a.row_map = nullptr;
  return cudaSuccess;
}

// Schedule of the scoring launch: one W pass per batch and a light epilogue.
//
// Row-tile pairs (kPrecBf16x2): each work item is two row tiles against one W
// tile, so a W tile is streamed by half as many CTAs and every W k-slice in shared
// memory feeds two row tiles (a third fewer L2 reads per MMA), while every row
// still sees the MMA sequence and epilogue of the one-tile form.  A pair holds
// all of TMEM, so its epilogue is exposed once per item; that fixed cost weighs
// against MMAs that last 2 d / 16 K steps, so the pairs pay off at d >= 4096 for
// every even tile count, and below that only for batches of 2-4 row tiles (the
// bandwidth-bound knee).  Odd counts run one row tile per item (a lone last tile
// per W tile would hand some CTAs half the work of others).  Beyond one raster
// group the pairs' group at d = 4096 is 20 pairs (40 row tiles): the pairs keep
// twice as many W tiles in flight beside the group's y panel, and a 48-tile
// group let the panel spill (11.2 GB of DRAM reads per 32768-row launch against
// 9.3 GB with 40 tiles).  When several work items share a W tile inside one
// raster group (batches of up to one group), the CTA on the tile's first item
// prefetches the tile's W k-blocks into L2 kLeaderPrefetch k-blocks ahead of its
// own loads, so that the other CTAs on the tile, which request the same
// k-blocks, are not held to one ring's depth of DRAM requests in flight.
// Measured on GB300 (V = 151936, whole calls; builds or variants side by side in
// one process, alternating in random order, bitwise equal outputs):
//  * d = 4096 within one raster group, against the previous schedule (pairs for
//    even counts and for odd counts whose pair count is coprime with the CTA
//    count, no prefetch) and with the epilogue's overlapped TMEM loads: 448 rows
//    411 -> 395 us, 512 rows 429 -> 416, 513 rows 533 -> 516, 640 rows 546 ->
//    531, 768 rows 613 -> 602, 1024 rows 794 -> 779, 2048 rows 1523 -> 1496; 128,
//    256, 384, 1408 and 4096 rows within 0.3%.  Prefetching 8 k-blocks ahead was
//    no better than 4; prefetching where each CTA streams its own W tile (64-256
//    rows: +5-10%) or in batches of several raster groups (32768 rows: +10%) was
//    slower;
//  * d = 4096 beyond one raster group, one tile per item -> pairs in groups of
//    24 / 20 / 16 pairs (20 back-to-back calls per sample, 8 rounds): 32768 rows
//    23575 -> 23377 / 23061 / 23226 us (28 pairs: 23987), 16384 rows 11766 ->
//    11571 / 11538 us;
//  * d = 5120: one tile per item -> pairs, 256-4096 rows 311 -> 285, 574 -> 506,
//    1107 -> 950, 2061 -> 1927, 3854 -> 3786 us; 131072 rows 118.6 -> 115.9 ms
//    (groups of 18 pairs);
//  * d = 2048: one tile per item -> pairs, 256 rows 130 -> 130 us, 512 rows 231
//    -> 224, 768 rows 309 -> 329, 1024 rows 440 -> 429, 2048 rows 776 -> 839,
//    4096 rows 1456 -> 1653, 6144 rows 2254 -> 2373, 8192 rows 2917 -> 3041-3092.
constexpr int kLeaderPrefetch = 4;

static bool plan_scoring_schedule(GemmArgs& a) {
  const bool one_group = a.num_m <= a.group_m;
  const bool long_k = a.d >= 4096;
  const bool pairs = a.num_m >= 2 && a.num_m % 2 == 0 && (long_k || a.num_m <= 4);
  if (pairs) {
    a.num_m /= 2;  // work items along M: row-tile pairs
    a.group_m = (!one_group && a.d <= 4096) ? 20 : (a.group_m + 1) / 2;
    a.num_tiles = static_cast<int64_t>(a.num_m) * a.num_n;
  }
  a.w_prefetch = (one_group && a.num_m >= 2) ? kLeaderPrefetch : 0;
  return pairs;
}

// W holds V vocabulary rows whose global ids start at v0 (a vocabulary shard when
// v0 > 0 or V is not the whole vocabulary); records are written per local tile.
cudaError_t launch_lmhead_lse_shard(const void* y, const void* W, const int32_t* ids, int64_t T,
                                    int d, int V, int v0, float temperature, void* part,
                                    float* tgt, int* status, cudaStream_t stream, int num_sms) {
  CUtensorMap map_y, map_w;
  GemmArgs a;
  cudaError_t e = make_args(a, map_y, map_w, y, W, ids, T, d, V, v0, temperature, status);
  if (e != cudaSuccess) return e;
  a.part = static_cast<float4*>(part);
  a.tgt = tgt;
  // Programmatic overlap with the RMSNorm kernel pays off while all row tiles
  // fit one raster group (decode-sized and mid-sized batches: measured 10-200 us
  // faster up to 4096 rows); beyond that the early-launched grid ran slower
  // (3 ms at 32768 rows), so larger batches are launched in stream order.  The
  // arithmetic is identical either way.
  const bool programmatic = a.num_m <= a.group_m;
  if (plan_scoring_schedule(a))
    return launch_gemm<0, kPrecBf16x2>(map_y, map_w, map_y, map_w, a, stream, num_sms,
                                       programmatic);
  return launch_gemm<0, kPrecBf16>(map_y, map_w, map_y, map_w, a, stream, num_sms, programmatic);
}

// FP8 head: y8 e4m3 [rows_padded(T), d] with per-row scales sy, W8 e4m3 [V, d]
// with per-row scales sw (d a multiple of 128).
cudaError_t launch_lmhead_lse_fp8(const void* y8, const float* sy, const void* W8,
                                  const float* sw, const int32_t* ids, int64_t T, int d, int V,
                                  float temperature, void* part, float* tgt, int* status,
                                  cudaStream_t stream, int num_sms) {
  CUtensorMap map_y, map_w;
  GemmArgs a;
  cudaError_t e =
      make_args(a, map_y, map_w, y8, W8, ids, T, d, V, 0, temperature, status, kPrecE4m3);
  if (e != cudaSuccess) return e;
  a.part = static_cast<float4*>(part);
  a.tgt = tgt;
  a.sy = sy;
  a.sw = sw;
  return launch_gemm<0, kPrecE4m3>(map_y, map_w, map_y, map_w, a, stream, num_sms, false);
}

// FP32 head: y and W in fp32, each split into a tf32 part and its fp32 remainder:
// y_big / y_small [rows_padded(T), d], W_big / W_small [V, d] (d a multiple of 32).
cudaError_t launch_lmhead_lse_tf32x3(const float* y_big, const float* y_small, const float* W_big,
                                     const float* W_small, const int32_t* ids, int64_t T, int d,
                                     int V, float temperature, void* part, float* tgt,
                                     int* status, cudaStream_t stream, int num_sms) {
  CUtensorMap map_y, map_w, map_y2, map_w2;
  GemmArgs a;
  cudaError_t e = make_args(a, map_y, map_w, y_big, W_big, ids, T, d, V, 0, temperature, status,
                            kPrecTf32x3);
  if (e != cudaSuccess) return e;
  if (!make_kmajor_map(&map_y2, y_small, static_cast<uint64_t>(rows_padded(T)),
                       static_cast<uint64_t>(d), kBM, kPrecTf32x3) ||
      !make_kmajor_map(&map_w2, W_small, static_cast<uint64_t>(V), static_cast<uint64_t>(d), kBN,
                       kPrecTf32x3))
    return cudaErrorInvalidValue;
  a.part = static_cast<float4*>(part);
  a.tgt = tgt;
  return launch_gemm<0, kPrecTf32x3>(map_y, map_w, map_y2, map_w2, a, stream, num_sms, false);
}

// Candidate collection pass of the processed score: logits >= thr[row] are
// appended to cand[row][0 .. cap) with cnt[row] counting them (counts above cap
// mean the row overflowed).  Launched without programmatic overlap: the
// thresholds and zeroed counters come from the kernel just before it.
// With dyn_T set, y holds up to T gathered rows of which only the first *dyn_T
// are live; row r's candidates and threshold belong to row row_map[r].  Row tiles
// are then scheduled one after another (raster groups of one row tile), so the
// few live ones spread over all CTAs.
cudaError_t launch_lmhead_collect(const void* y, const void* W, const int32_t* ids, int64_t T,
                                  int d, int V, float temperature, const float* thr, int* cnt,
                                  void* cand, int cap, const int* dyn_T, const int* row_map,
                                  int* status, cudaStream_t stream, int num_sms) {
  CUtensorMap map_y, map_w;
  GemmArgs a;
  cudaError_t e = make_args(a, map_y, map_w, y, W, ids, T, d, V, 0, temperature, status);
  if (e != cudaSuccess) return e;
  a.thr = thr;
  a.cnt = cnt;
  a.cand = static_cast<uint2*>(cand);
  a.cap = cap;
  a.dyn_T = dyn_T;
  a.row_map = row_map;
  if (dyn_T != nullptr) a.group_m = 1;
  return launch_gemm<1, kPrecBf16>(map_y, map_w, map_y, map_w, a, stream, num_sms, false);
}

// Processed score, pass 1: the four largest logits of every (row, 256-column
// tile) with their ids, as Top4 records [ceil(T/32)][num_n][32].
cudaError_t launch_lmhead_top4(const void* y, const void* W, const int32_t* ids, int64_t T, int d,
                               int V, void* top4, int* status, cudaStream_t stream, int num_sms) {
  CUtensorMap map_y, map_w;
  GemmArgs a;
  cudaError_t e = make_args(a, map_y, map_w, y, W, ids, T, d, V, 0, 1.0f, status);
  if (e != cudaSuccess) return e;
  a.top4 = top4;
  // One row tile per item at every size: the top-4 epilogue (an insertion per
  // logit) is heavy enough that a row-tile pair's exposed epilogue costs more than
  // the shared W saves (GB300, processed score k = 50, p = 0.95, d = 4096, same-
  // process A/B, bitwise equal outputs: 256-32768 rows 5-25% slower with pairs,
  // e.g. 4096 rows 3.16 -> 3.94 ms).  The leader's L2 prefetch of W is kept for
  // batches within one raster group, as in the scoring launch.
  a.w_prefetch = (a.num_m <= a.group_m && a.num_m >= 2) ? kLeaderPrefetch : 0;
  return launch_gemm<4, kPrecBf16>(map_y, map_w, map_y, map_w, a, stream, num_sms, false);
}

// Backward, step 1: recompute z = y . W^T and write G = dL/dz (bf16) as
// gz [rows_padded(T)][ldg] (rows past T written as zeros).
cudaError_t launch_logit_grad(const void* y, const void* W, const int32_t* ids, const float* lse,
                              const float* gup, int64_t T, int d, int V, float temperature,
                              uint16_t* gz, int64_t ldg, int* status, cudaStream_t stream,
                              int num_sms) {
  CUtensorMap map_y, map_w;
  GemmArgs a;
  cudaError_t e = make_args(a, map_y, map_w, y, W, ids, T, d, V, 0, temperature, status);
  if (e != cudaSuccess) return e;
  a.lse = lse;
  a.gup = gup;
  a.gz = gz;
  a.ldg = ldg;
  return launch_gemm<2, kPrecBf16>(map_y, map_w, map_y, map_w, a, stream, num_sms, false);
}

// Backward, steps 2 and 3: C [M][N] (+)= A . B^T, fp32 C with row stride ldc,
// N a multiple of 32.  A (M x K) is bf16 K-major [M][lda] (a_mn = 0; rows_a >= M
// rows readable) or MN-major [K][lda] (a_mn = 1; M contiguous); likewise B (N x
// K) is [N][ldb] (b_mn = 0) or [K][ldb] (b_mn = 1).  The MN-major forms let the
// products read G, W and y where they lie, with no transposed copies.
cudaError_t launch_gemm_store(const void* A, int64_t rows_a, int64_t lda, int a_mn, const void* B,
                              int N, int64_t ldb, int b_mn, int64_t K, int64_t M, float* C,
                              int64_t ldc, int accumulate, int* status, cudaStream_t stream,
                              int num_sms) {
  CUtensorMap map_a, map_b;
  const bool ok_a = a_mn ? make_bf16_mn_map(&map_a, A, static_cast<uint64_t>(M),
                                            static_cast<uint64_t>(K), static_cast<uint64_t>(lda))
                         : make_bf16_map(&map_a, A, static_cast<uint64_t>(rows_a),
                                         static_cast<uint64_t>(K), static_cast<uint64_t>(lda), kBM);
  const bool ok_b = b_mn ? make_bf16_mn_map(&map_b, B, static_cast<uint64_t>(N),
                                            static_cast<uint64_t>(K), static_cast<uint64_t>(ldb))
                         : make_bf16_map(&map_b, B, static_cast<uint64_t>(N),
                                         static_cast<uint64_t>(K), static_cast<uint64_t>(ldb), kBN);
  if (!ok_a || !ok_b) return cudaErrorInvalidValue;
  GemmArgs a = {};
  a.T = M;
  a.v0 = 0;
  a.v_end = N;
  a.d = static_cast<int>(K < INT32_MAX ? K : INT32_MAX);
  a.num_m = static_cast<int>((M + kBM - 1) / kBM);
  a.num_n = (N + kBN - 1) / kBN;
  a.num_kb = static_cast<int>((K + kBK - 1) / kBK);
  // Raster groups of 2 row tiles: with K = V or K = T the operand panels of a
  // tile (128 or 256 rows x K) are megabytes long; whole backward calls at
  // T = 32768, d = 4096 with one row tile per item (groups for G.W / G^T.y): 2/2
  // 76.6-76.8 ms, 1/2 76.9, 2/1 77.1, 4/2 77.3, 2/16 77.5, 16/2 78.2, 16/16 79.2
  // (48: 82.1 before the products read G and W in place).
  a.group_m = 2;
  a.num_tiles = static_cast<int64_t>(a.num_m) * a.num_n;
  a.k2 = 0.f;
  a.inv_temp = 0.f;
  a.ids = nullptr;
  a.status = status;
  a.c = C;
  a.ldc = ldc;
  a.accumulate = accumulate;
  a.a_mn = a_mn;
  a.b_mn = b_mn;
  a.wait_limit_ns = kWaitLimitNs;
  a.stall_producer = 0;
  // Two or more row tiles: work items are row-tile pairs sharing each B k-slice in
  // shared memory (kPrecBf16x2), so the two tiles advance along K in lockstep and
  // B is read from L2 once for both.  With K = V or K = T a tile's MMAs run for
  // hundreds of microseconds, so the single accumulator buffer of a pair costs
  // well under 1% in epilogue time.  The raster group is then one pair (the same
  // 2 row tiles).  Whole backward at T = 32768, d = 4096: 76.4 -> 69.8 ms.
  if (a.num_m >= 2) {
    a.num_m = (a.num_m + 1) / 2;
    a.group_m = 1;
    a.num_tiles = static_cast<int64_t>(a.num_m) * a.num_n;
    return launch_gemm<3, kPrecBf16x2>(map_a, map_b, map_a, map_b, a, stream, num_sms, false);
  }
  return launch_gemm<3, kPrecBf16>(map_a, map_b, map_a, map_b, a, stream, num_sms, false);
}

// Self-test of the bounded waits: the scoring kernel with its producer stalled (no
// load is ever issued), so the MMA warp's first wait on a full stage and the
// epilogue's wait on the accumulator run out after limit_ns; every CTA records
// TIM_ERR_TIMEOUT, winds down and frees its TMEM.  y, W and ids must be valid
// device memory of the stated shapes (never read by the tensor cores).
cudaError_t launch_wait_selftest(const void* y, const void* W, const int32_t* ids, int64_t T,
                                 int d, int V, void* part, float* tgt, int* status,
                                 uint64_t limit_ns, cudaStream_t stream, int num_sms) {
  CUtensorMap map_y, map_w;
  GemmArgs a;
  cudaError_t e = make_args(a, map_y, map_w, y, W, ids, T, d, V, 0, 1.0f, status);
  if (e != cudaSuccess) return e;
  a.part = static_cast<float4*>(part);
  a.tgt = tgt;
  a.wait_limit_ns = limit_ns;
  a.stall_producer = 1;
  return launch_gemm<0, kPrecBf16>(map_y, map_w, map_y, map_w, a, stream, num_sms, false);
}

// Places the scoring path's two kernel forms (one row tile or a row-tile pair per
// work item) on the current device now rather than at their first launch: the
// CUDA runtime loads kernels lazily, and loading one takes device memory.
cudaError_t load_scoring_gemm_kernels() {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, lmhead_lse_kernel<0, kPrecBf16>);
  if (e != cudaSuccess) return e;
  return cudaFuncGetAttributes(&attr, lmhead_lse_kernel<0, kPrecBf16x2>);
}

cudaError_t launch_lmhead_lse(const void* y, const void* W, const int32_t* ids, int64_t T,
                              int d, int V, float temperature, void* part, float* tgt,
                              int* status, cudaStream_t stream, int num_sms) {
  return launch_lmhead_lse_shard(y, W, ids, T, d, V, 0, temperature, part, tgt, status, stream,
                                 num_sms);
}

}  // namespace tim
