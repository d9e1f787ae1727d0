// Shared device helpers for the sm_103a kernels: status word, workspace
// layout, bounded mbarrier waits, TMA, and tcgen05 (UMMA / TMEM) wrappers.
// All inline PTX here is hand-written from the PTX ISA's instruction
// descriptions (mbarrier, cp.async.bulk.tensor, tcgen05.*).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tim.h"

namespace tim {

// ---------------------------------------------------------------------------
// Tiling of the LM-head GEMM.  One shape for every T: the K-reduction order of
// a logit never depends on the batch.
constexpr int kBM = 128;          // rows (tokens) per tile = UMMA M
constexpr int kBN = 256;          // vocabulary columns per tile = UMMA N = leaf tile width
constexpr int kBK = 64;           // K elements per stage (= one 128-byte swizzle row of bf16)
constexpr int kUmmaK = 16;        // K per tcgen05.mma (kind::f16)
constexpr int kStages = 4;        // smem pipeline depth
constexpr int kABytes = kBM * kBK * 2;   // 16 KiB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KiB
constexpr int kEpiWarps = 4;             // one epilogue warp per TMEM lane quadrant
constexpr int kTmemCols = 512;           // two 256-column fp32 accumulators
constexpr int kRowGroup = 32;            // rows per partial-record group

// Partial-record layout: [ceil(T/32)][n_tiles][32] x float4
//   .x = max over the tile of z * log2(e)/tau  (base-2 domain)
//   .y = sum over the tile of 2^(z*log2(e)/tau - .x)
//   .z = largest raw logit z in the tile
//   .w = its vocabulary id (int bits; lowest id on ties)

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 1024-byte aligned).
struct WsLayout {
  size_t status_off;   // int32 status word (+ padding)
  size_t y_off;        // bf16 [rows_padded(T), d]; rows >= T are zero
  size_t part_off;     // float4 [ceil(T/32)][n_tiles][32]
  size_t tgt_off;      // float32 [T]
  size_t total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// y is stored with whole 128-row tiles (zero rows past T) so the LM-head TMA
// never reads outside the tensor.
__host__ __device__ inline int64_t rows_padded(int64_t T) { return (T + kBM - 1) / kBM * kBM; }

__host__ inline WsLayout logprob_layout(int64_t T, int32_t d, int32_t V) {
  WsLayout L;
  const size_t n_tiles = ((size_t)V + kBN - 1) / kBN;
  const size_t groups = ((size_t)T + kRowGroup - 1) / kRowGroup;
  L.status_off = 0;
  L.y_off = 1024;
  L.part_off = align_up(L.y_off + (size_t)rows_padded(T) * (size_t)d * 2, 1024);
  L.tgt_off = align_up(L.part_off + groups * n_tiles * kRowGroup * 16, 1024);
  L.total = align_up(L.tgt_off + (size_t)T * 4, 1024);
  return L;
}

// ---------------------------------------------------------------------------
// Status word: first error wins.
__device__ __forceinline__ void set_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

// Bounded waits: a wait gives up after this many nanoseconds of wall time,
// records TIM_ERR_TIMEOUT and lets the kernel wind down.
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;   // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Test the phase; if it is not complete the thread may be suspended until it
// completes or kSuspendHintNs passes (fewer spinning warps compete for issue
// slots with the MMA-issuing thread and the epilogue).
constexpr uint32_t kSuspendHintNs = 20000u;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if the
// shared abort flag was raised or the time limit passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA: 2-D tiled bulk tensor load global -> shared, completion counted in bytes
// on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// L2 prefetch of one 2-D tile of a tensor map (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, accumulators in tensor memory)
__device__ __forceinline__ void tmem_alloc(uint32_t* holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(holder_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row atoms of 1024 bytes.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4 (unused for this layout; 1)
//   bits 32-45 stride-dimension byte offset >> 4 (1024 bytes between 8-row atoms)
//   bits 46-48 fixed 0b001
//   bits 61-63 swizzle mode (2 = 128-byte swizzle)
// Stepping K by 16 elements inside the 128-byte row adds 32 bytes to the start.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  desc |= static_cast<uint64_t>(1u) << 16;
  desc |= static_cast<uint64_t>(1024u >> 4) << 32;
  desc |= static_cast<uint64_t>(1u) << 46;
  desc |= static_cast<uint64_t>(2u) << 61;
  return desc;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4: D fp32, A and B e4m3 (format code 0),
// both K-major; same M/N fields as above.
__host__ __device__ constexpr uint32_t umma_idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::tf32: D fp32, A and B tf32 (format code 2),
// both K-major; same M/N fields as above.
__host__ __device__ constexpr uint32_t umma_idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D += A * B with tf32 operands (fp32 storage, K = 8 per instruction), fp32
// accumulation.
__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D += A * B with e4m3 operands (K = 32 per instruction), fp32 accumulation.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Per-sequence work partition shared by the compare and diagnostics kernels:
// sequence j is cut into P_j = clamp(ceil(len_j / 256), 1, 256) contiguous parts
// (1 for invalid offsets), numbered globally from base[j]; base[n_seq] = total.
// P_j depends only on the sequence's own length, so its partial sums -- and the
// fp64 statistics folded from them -- do not depend on the batch.
constexpr int kSeqTokensPerPart = 256;
constexpr int kSeqMaxParts = 256;

__host__ __device__ inline int seq_parts(int64_t s, int64_t e, int64_t T) {
  if (!(s >= 0 && s <= e && e <= T)) return 1;
  int64_t P = (e - s + kSeqTokensPerPart - 1) / kSeqTokensPerPart;
  if (P < 1) P = 1;
  if (P > kSeqMaxParts) P = kSeqMaxParts;
  return static_cast<int>(P);
}

// Upper bound of the total part count (sum_j ceil(len_j / 256) <= T / 256 + n_seq).
__host__ inline int64_t seq_parts_bound(int64_t T, int n_seq) {
  return (T + kSeqTokensPerPart - 1) / kSeqTokensPerPart + n_seq;
}

// The sequence whose parts include global part index b: the largest j with
// base[j] <= b (base ascending, n_seq + 1 entries, base[0] = 0).
__device__ __forceinline__ int part_sequence(const int* base, int n_seq, int b) {
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldcg(base + mid) <= b) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The four largest logits of one (row, 256-column tile): values descending and
// their vocabulary ids (equal values: the lower id first); -inf / -1 past the
// tile.  Written by the LM-head kernel in top-4 mode, read by the processed
// score's candidate kernel.  Layout [ceil(T/32)][n_tiles][32].
struct Top4Rec {
  float v[4];
  int32_t id[4];
};

// L2 policy for data written once and read back only much later (streams that
// would otherwise evict the operands the tensor cores are re-reading).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void st_global_v4_hint(void* ptr, const uint4& v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void st_global_u16_hint(void* ptr, uint16_t v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(ptr), "h"(v), "l"(policy)
               : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape,
// x32 repetitions) and wait for the load in the same asm block, so no use of
// the registers can be scheduled before the data is there.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// The same load without its wait: the registers are written asynchronously and
// must not be read before tmem_ld_wait on them.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Wait for this thread's outstanding tcgen05.ld.  The registers of the load are
// passed through the wait, so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now / wait until the previous kernel's memory is visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 2^x with the hardware approximation (MUFU.EX2), flush-to-zero.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace tim
