// C ABI of libtim: argument validation, workspace layout, status handling and
// kernel launches on the caller's stream.  See include/tim.h for the contract.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "tim_common.cuh"

namespace tim {
cudaError_t launch_rmsnorm_rows(const void* hidden, const void* gamma, int64_t T, int d, float eps,
                                void* y, int* status, cudaStream_t stream);
cudaError_t launch_lmhead_lse(const void* y, const void* W, const int32_t* ids, int64_t T, int d,
                              int V, float temperature, void* part, float* tgt, int* status,
                              cudaStream_t stream, int num_sms);
cudaError_t launch_lse_finalize(const void* part, const float* tgt, const int32_t* ids, int64_t T,
                                int V, float* out_lp, float* out_lse, int32_t* out_top1,
                                int* status, cudaStream_t stream);
cudaError_t launch_seg_compare(const float* A, const float* B, const float* C,
                               const int64_t* offs, int n_seq, const uint8_t* mask, int64_t T,
                               float tis_cap, tim_seq_stats* out, float* tis_w, void* workspace,
                               cudaStream_t stream);
size_t compare_workspace_bytes(int64_t T, int n_seq);
cudaError_t launch_lmhead_lse_shard(const void* y, const void* W, const int32_t* ids, int64_t T,
                                    int d, int V, int v0, float temperature, void* part,
                                    float* tgt, int* status, cudaStream_t stream, int num_sms);
void vocab_shard_range(int V, int G, int g, int* v0, int* v_len);
cudaError_t launch_quantize_rows_e4m3(const void* x, int64_t rows, int K, void* codes,
                                      float* scales, cudaStream_t stream);
cudaError_t launch_rmsnorm_rows_split(const void* hidden, const void* gamma, int64_t T, int d,
                                      float eps, float* ybig, float* ysmall, int* status,
                                      cudaStream_t stream);
cudaError_t launch_split_tf32(const float* x, int64_t n, float* big, float* small,
                              cudaStream_t stream, int num_sms);
cudaError_t launch_lmhead_lse_tf32x3(const float* y_big, const float* y_small, const float* W_big,
                                     const float* W_small, const int32_t* ids, int64_t T, int d,
                                     int V, float temperature, void* part, float* tgt,
                                     int* status, cudaStream_t stream, int num_sms);
cudaError_t launch_logit_grad(const void* y, const void* W, const int32_t* ids, const float* lse,
                              const float* gup, int64_t T, int d, int V, float temperature,
                              uint16_t* gz, int64_t ldg, int* status, cudaStream_t stream,
                              int num_sms);
cudaError_t launch_gemm_store(const void* A, int64_t rows_a, int64_t lda, int a_mn, const void* B,
                              int N, int64_t ldb, int b_mn, int64_t K, int64_t M, float* C,
                              int64_t ldc, int accumulate, int* status, cudaStream_t stream,
                              int num_sms);
cudaError_t launch_wait_selftest(const void* y, const void* W, const int32_t* ids, int64_t T,
                                 int d, int V, void* part, float* tgt, int* status,
                                 uint64_t limit_ns, cudaStream_t stream, int num_sms);
int rmsnorm_backward_chunks(int64_t T);
cudaError_t launch_rmsnorm_backward(const void* hidden, const void* gamma, const float* dy,
                                    int64_t T, int d, float eps, float* dh, float* dgamma,
                                    int accumulate, float* rstd, float* partial, int* status,
                                    cudaStream_t stream);
cudaError_t launch_lmhead_lse_fp8(const void* y8, const float* sy, const void* W8,
                                  const float* sw, const int32_t* ids, int64_t T, int d, int V,
                                  float temperature, void* part, float* tgt, int* status,
                                  cudaStream_t stream, int num_sms);
cudaError_t launch_lmhead_collect(const void* y, const void* W, const int32_t* ids, int64_t T,
                                  int d, int V, float temperature, const float* thr, int* cnt,
                                  void* cand, int cap, const int* dyn_T, const int* row_map,
                                  int* status, cudaStream_t stream, int num_sms);
cudaError_t launch_lmhead_top4(const void* y, const void* W, const int32_t* ids, int64_t T, int d,
                               int V, void* top4, int* status, cudaStream_t stream, int num_sms);
cudaError_t launch_topk_candidates(const void* top4, int64_t T, int V, int k, float* thr,
                                   int* cnt, void* cand, int cap, int* fb_count, int* fb_rows,
                                   cudaStream_t stream);
cudaError_t launch_gather_rows(const void* y, const int* fb_rows, const int* fb_count, int64_t T,
                               int d, void* y_fb, cudaStream_t stream, int num_sms);
cudaError_t launch_topk_finalize(const void* cand, const int* cnt, const int32_t* ids, int64_t T,
                                 int V, int k, float top_p, float temperature, int cap,
                                 float* out_lp, float* out_lse, int32_t* out_kept,
                                 int32_t* head_ids, float* head_lp, int* status,
                                 cudaStream_t stream);
cudaError_t launch_shard_reduce(const void* part, const float* tgt, int64_t T, int V, int G, int g,
                                int v_len, void* out_rec, float* out_tgt, cudaStream_t stream);
cudaError_t launch_merge_shards(const void* recs, const float* tgts, const int32_t* ids, int64_t T,
                                int V, int G, float* out_lp, float* out_lse, int32_t* out_top1,
                                int* status, cudaStream_t stream);
cudaError_t launch_seg_diag(const float* A, const float* B, const float* C, const int32_t* tA,
                            const int32_t* tB, const int32_t* tC, const int64_t* offs, int n_seq,
                            const uint8_t* mask, int64_t T, float tis_cap, float mis_lo,
                            float mis_hi, tim_seq_diag* out, void* workspace,
                            cudaStream_t stream);
size_t diag_workspace_bytes(int64_t T, int n_seq);

namespace {

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

tim_status check_shape(int64_t T, int32_t d, int32_t V) {
  if (T < 1 || T > INT32_MAX) return TIM_ERR_SHAPE;
  if (d < 64 || d > 65536 || (d % 64) != 0) return TIM_ERR_SHAPE;
  if (V < 1 || V > INT32_MAX - 256) return TIM_ERR_SHAPE;
  return TIM_OK;
}

tim_status check_scalars(float temperature, float eps) {
  if (!(std::isfinite(temperature) && temperature > 0.f)) return TIM_ERR_INVALID_ARG;
  if (!(std::isfinite(eps) && eps >= 0.f)) return TIM_ERR_INVALID_ARG;
  return TIM_OK;
}

tim_status check_workspace(const void* ws, size_t bytes, size_t need) {
  if (ws == nullptr || !aligned(ws, 256) || bytes < need) return TIM_ERR_WORKSPACE;
  return TIM_OK;
}

// The current device must be an sm_103 part.  Returns its SM count.
tim_status check_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TIM_ERR_CUDA;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return TIM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return TIM_ERR_UNSUPPORTED_DEVICE;
  if (num_sms != nullptr) *num_sms = sms;
  return TIM_OK;
}

inline tim_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TIM_OK : TIM_ERR_CUDA; }

struct Ptrs {
  int* status;
  void* y;
  void* part;
  float* tgt;
};

Ptrs logprob_ptrs(void* ws, int64_t T, int32_t d, int32_t V) {
  const WsLayout L = logprob_layout(T, d, V);
  uint8_t* b = static_cast<uint8_t*>(ws);
  return Ptrs{reinterpret_cast<int*>(b + L.status_off), b + L.y_off, b + L.part_off,
              reinterpret_cast<float*>(b + L.tgt_off)};
}

tim_status validate_logprob_common(int64_t T, int32_t d, int32_t V, float temperature,
                                   float eps, const void* ws, size_t ws_bytes) {
  tim_status s = check_shape(T, d, V);
  if (s != TIM_OK) return s;
  if ((s = check_scalars(temperature, eps)) != TIM_OK) return s;
  return check_workspace(ws, ws_bytes, logprob_layout(T, d, V).total);
}

// Processed-score workspace: the scoring workspace, then thresholds [T],
// candidate counters [T], candidate slots [T][TIM_PROCESSED_CAPACITY], top-4
// records [ceil(T/32) * 32][n_tiles], the fallback row count and list [T], and
// the gathered fallback rows of y [rows_padded(T), d].
struct ProcLayout {
  WsLayout base;
  size_t thr_off, cnt_off, cand_off, top4_off, fbn_off, fbrows_off, yfb_off, total;
};
ProcLayout processed_layout(int64_t T, int32_t d, int32_t V) {
  ProcLayout P;
  P.base = logprob_layout(T, d, V);
  const size_t n_tiles = (static_cast<size_t>(V) + kBN - 1) / kBN;
  const size_t t32 = (static_cast<size_t>(T) + 31) / 32 * 32;
  P.thr_off = align_up(P.base.total, 1024);
  P.cnt_off = align_up(P.thr_off + static_cast<size_t>(T) * 4, 1024);
  P.cand_off = align_up(P.cnt_off + static_cast<size_t>(T) * 4, 1024);
  P.top4_off = align_up(P.cand_off + static_cast<size_t>(T) * TIM_PROCESSED_CAPACITY * 8, 1024);
  P.fbn_off = align_up(P.top4_off + t32 * n_tiles * sizeof(Top4Rec), 1024);
  P.fbrows_off = P.fbn_off + 256;
  P.yfb_off = align_up(P.fbrows_off + static_cast<size_t>(T) * 4, 1024);
  P.total = align_up(P.yfb_off + static_cast<size_t>(rows_padded(T)) * d * 2, 1024);
  return P;
}

// FP8 workspace: the scoring workspace, then y codes [rows_padded(T), d] and
// their per-row scales [rows_padded(T)].
struct Fp8Layout {
  WsLayout base;
  size_t y8_off, sy_off, total;
};
Fp8Layout fp8_layout(int64_t T, int32_t d, int32_t V) {
  Fp8Layout F;
  F.base = logprob_layout(T, d, V);
  const size_t rows = static_cast<size_t>(rows_padded(T));
  F.y8_off = align_up(F.base.total, 1024);
  F.sy_off = align_up(F.y8_off + rows * static_cast<size_t>(d), 1024);
  F.total = align_up(F.sy_off + rows * 4, 1024);
  return F;
}

// FP32 workspace: the scoring workspace, then the tf32 part and the remainder of
// y, fp32 [rows_padded(T), d] each.
struct Fp32Layout {
  WsLayout base;
  size_t ybig_off, ysmall_off, total;
};
Fp32Layout fp32_layout(int64_t T, int32_t d, int32_t V) {
  Fp32Layout F;
  F.base = logprob_layout(T, d, V);
  const size_t n = static_cast<size_t>(rows_padded(T)) * static_cast<size_t>(d) * 4;
  F.ybig_off = align_up(F.base.total, 1024);
  F.ysmall_off = align_up(F.ybig_off + n, 1024);
  F.total = align_up(F.ysmall_off + n, 1024);
  return F;
}

// Backward workspace: status | y bf16 [Tp, d] | y^T [d, Tp] | W^T [d, Vp] |
// G [Tp, Vp] | G^T [Vp, Tp], with Tp = rows_padded(T) and Vp = V rounded up to 64.
// Backward workspace: status | y bf16 [Tp][d] | G bf16 [Tp][Vp].
struct BwdLayout {
  int64_t Tp, Vp;
  size_t status_off, y_off, g_off, total;
};
BwdLayout backward_layout(int64_t T, int32_t d, int32_t V) {
  BwdLayout B;
  B.Tp = rows_padded(T);
  B.Vp = (static_cast<int64_t>(V) + 63) / 64 * 64;
  const size_t dd = static_cast<size_t>(d);
  B.status_off = 0;
  B.y_off = 1024;
  B.g_off = align_up(B.y_off + static_cast<size_t>(B.Tp) * dd * 2, 1024);
  B.total = align_up(B.g_off + static_cast<size_t>(B.Tp) * static_cast<size_t>(B.Vp) * 2, 1024);
  return B;
}

bool valid_shard(int32_t G, int32_t g) {
  return (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) && g >= 0 && g < G;
}

}  // namespace
}  // namespace tim

using namespace tim;

extern "C" {

const char* tim_status_string(tim_status s) {
  switch (s) {
    case TIM_OK: return "TIM_OK";
    case TIM_ERR_INVALID_ARG: return "TIM_ERR_INVALID_ARG";
    case TIM_ERR_SHAPE: return "TIM_ERR_SHAPE";
    case TIM_ERR_TOKEN_RANGE: return "TIM_ERR_TOKEN_RANGE";
    case TIM_ERR_NONFINITE: return "TIM_ERR_NONFINITE";
    case TIM_ERR_EMPTY_SEQUENCE: return "TIM_ERR_EMPTY_SEQUENCE";
    case TIM_ERR_BAD_MASK: return "TIM_ERR_BAD_MASK";
    case TIM_ERR_WORKSPACE: return "TIM_ERR_WORKSPACE";
    case TIM_ERR_CUDA: return "TIM_ERR_CUDA";
    case TIM_ERR_TIMEOUT: return "TIM_ERR_TIMEOUT";
    case TIM_ERR_UNSUPPORTED_DEVICE: return "TIM_ERR_UNSUPPORTED_DEVICE";
    case TIM_ERR_CAPACITY: return "TIM_ERR_CAPACITY";
  }
  return "TIM_ERR_UNKNOWN";
}

int32_t tim_abi_version(void) { return TIM_ABI_VERSION; }

tim_status tim_workspace_init(void* workspace, size_t workspace_bytes, tim_stream_t stream) {
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < 256)
    return TIM_ERR_WORKSPACE;
  return from_cuda(
      cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

tim_status tim_status_sync(void* workspace, tim_stream_t stream) {
  if (workspace == nullptr) return TIM_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TIM_ERR_CUDA;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TIM_ERR_CUDA;
  if (v != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return TIM_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return TIM_ERR_CUDA;
  }
  return static_cast<tim_status>(v);
}

size_t tim_logprob_workspace_size(int64_t T, int32_t d, int32_t V) {
  if (check_shape(T, d, V) != TIM_OK) return 0;
  return logprob_layout(T, d, V).total;
}

tim_status tim_rmsnorm_rows(const void* hidden, const void* gamma, int64_t T, int32_t d,
                            int32_t V, float eps, void* workspace, size_t workspace_bytes,
                            tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr) return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16)) return TIM_ERR_INVALID_ARG;
  tim_status s = validate_logprob_common(T, d, V, 1.0f, eps, workspace, workspace_bytes);
  if (s != TIM_OK) return s;
  if ((s = check_device(nullptr)) != TIM_OK) return s;
  const Ptrs p = logprob_ptrs(workspace, T, d, V);
  return from_cuda(launch_rmsnorm_rows(hidden, gamma, T, d, eps, p.y, p.status,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

tim_status tim_lmhead_lse(const void* W, const int32_t* token_ids, int64_t T, int32_t d,
                          int32_t V, float temperature, void* workspace, size_t workspace_bytes,
                          tim_stream_t stream) {
  if (W == nullptr || token_ids == nullptr) return TIM_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(token_ids, 4)) return TIM_ERR_INVALID_ARG;
  tim_status s = validate_logprob_common(T, d, V, temperature, 0.f, workspace, workspace_bytes);
  if (s != TIM_OK) return s;
  int sms = 0;
  if ((s = check_device(&sms)) != TIM_OK) return s;
  const Ptrs p = logprob_ptrs(workspace, T, d, V);
  return from_cuda(launch_lmhead_lse(p.y, W, token_ids, T, d, V, temperature, p.part, p.tgt,
                                     p.status, reinterpret_cast<cudaStream_t>(stream), sms));
}

tim_status tim_lse_finalize(const int32_t* token_ids, int64_t T, int32_t d, int32_t V,
                            float temperature, float* out_logprob, float* out_lse,
                            int32_t* out_top1, void* workspace, size_t workspace_bytes,
                            tim_stream_t stream) {
  if (token_ids == nullptr || out_logprob == nullptr || out_lse == nullptr || out_top1 == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(token_ids, 4) || !aligned(out_logprob, 4) || !aligned(out_lse, 4) ||
      !aligned(out_top1, 4))
    return TIM_ERR_INVALID_ARG;
  tim_status s = validate_logprob_common(T, d, V, temperature, 0.f, workspace, workspace_bytes);
  if (s != TIM_OK) return s;
  if ((s = check_device(nullptr)) != TIM_OK) return s;
  const Ptrs p = logprob_ptrs(workspace, T, d, V);
  return from_cuda(launch_lse_finalize(p.part, p.tgt, token_ids, T, V, out_logprob, out_lse,
                                       out_top1, p.status,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

tim_status tim_logprob(const void* hidden, const void* gamma, const void* W,
                       const int32_t* token_ids, int64_t T, int32_t d, int32_t V,
                       float temperature, float eps, float* out_logprob, float* out_lse,
                       int32_t* out_top1, void* workspace, size_t workspace_bytes,
                       tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || W == nullptr || token_ids == nullptr ||
      out_logprob == nullptr || out_lse == nullptr || out_top1 == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16) || !aligned(W, 16) || !aligned(token_ids, 4) ||
      !aligned(out_logprob, 4) || !aligned(out_lse, 4) || !aligned(out_top1, 4))
    return TIM_ERR_INVALID_ARG;
  tim_status s = validate_logprob_common(T, d, V, temperature, eps, workspace, workspace_bytes);
  if (s != TIM_OK) return s;
  if ((s = tim_rmsnorm_rows(hidden, gamma, T, d, V, eps, workspace, workspace_bytes, stream)) !=
      TIM_OK)
    return s;
  if ((s = tim_lmhead_lse(W, token_ids, T, d, V, temperature, workspace, workspace_bytes,
                          stream)) != TIM_OK)
    return s;
  return tim_lse_finalize(token_ids, T, d, V, temperature, out_logprob, out_lse, out_top1,
                          workspace, workspace_bytes, stream);
}

size_t tim_compare_workspace_size(int64_t T, int32_t n_seq) {
  if (T < 1 || n_seq < 1) return 0;
  return compare_workspace_bytes(T, n_seq);
}

tim_status tim_compare(const float* lp_gen, const float* lp_replay, const float* lp_train,
                       const int64_t* seq_offsets, int32_t n_seq, const uint8_t* mask, int64_t T,
                       float tis_cap, tim_seq_stats* out_stats, float* out_tis_w,
                       void* workspace, size_t workspace_bytes, tim_stream_t stream) {
  if (lp_gen == nullptr || lp_replay == nullptr || lp_train == nullptr || seq_offsets == nullptr ||
      mask == nullptr || out_stats == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(lp_gen, 4) || !aligned(lp_replay, 4) || !aligned(lp_train, 4) ||
      !aligned(seq_offsets, 8) || !aligned(out_stats, 8) ||
      (out_tis_w != nullptr && !aligned(out_tis_w, 4)))
    return TIM_ERR_INVALID_ARG;
  if (T < 1 || T > INT32_MAX || n_seq < 1) return TIM_ERR_SHAPE;
  if (!(std::isfinite(tis_cap) && tis_cap > 0.f)) return TIM_ERR_INVALID_ARG;
  tim_status s = check_workspace(workspace, workspace_bytes, tim_compare_workspace_size(T, n_seq));
  if (s != TIM_OK) return s;
  if ((s = check_device(nullptr)) != TIM_OK) return s;
  return from_cuda(launch_seg_compare(lp_gen, lp_replay, lp_train, seq_offsets, n_seq, mask, T,
                                      tis_cap, out_stats, out_tis_w, workspace,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

tim_status tim_quantize_fp8_rows(const void* x, int64_t rows, int32_t K, void* codes,
                                 float* scales, tim_stream_t stream) {
  if (x == nullptr || codes == nullptr || scales == nullptr) return TIM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(scales, 4)) return TIM_ERR_INVALID_ARG;
  if (rows < 1 || rows > INT32_MAX || K < 16 || (K % 16) != 0) return TIM_ERR_SHAPE;
  tim_status s = check_device(nullptr);
  if (s != TIM_OK) return s;
  return from_cuda(launch_quantize_rows_e4m3(x, rows, K, codes, scales,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

size_t tim_logprob_fp8_workspace_size(int64_t T, int32_t d, int32_t V) {
  if (check_shape(T, d, V) != TIM_OK || (d % 128) != 0) return 0;
  return fp8_layout(T, d, V).total;
}

tim_status tim_logprob_fp8(const void* hidden, const void* gamma, const void* W_codes,
                           const float* W_scales, const int32_t* token_ids, int64_t T, int32_t d,
                           int32_t V, float temperature, float eps, float* out_logprob,
                           float* out_lse, int32_t* out_top1, void* workspace,
                           size_t workspace_bytes, tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || W_codes == nullptr || W_scales == nullptr ||
      token_ids == nullptr || out_logprob == nullptr || out_lse == nullptr ||
      out_top1 == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16) || !aligned(W_codes, 16) ||
      !aligned(W_scales, 4) || !aligned(token_ids, 4) || !aligned(out_logprob, 4) ||
      !aligned(out_lse, 4) || !aligned(out_top1, 4))
    return TIM_ERR_INVALID_ARG;
  tim_status s = check_shape(T, d, V);
  if (s != TIM_OK) return s;
  if ((d % 128) != 0) return TIM_ERR_SHAPE;
  if ((s = check_scalars(temperature, eps)) != TIM_OK) return s;
  const Fp8Layout F = fp8_layout(T, d, V);
  if ((s = check_workspace(workspace, workspace_bytes, F.total)) != TIM_OK) return s;
  int sms = 0;
  if ((s = check_device(&sms)) != TIM_OK) return s;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(b + F.base.status_off);
  void* y = b + F.base.y_off;
  void* part = b + F.base.part_off;
  float* tgt = reinterpret_cast<float*>(b + F.base.tgt_off);
  void* y8 = b + F.y8_off;
  float* sy = reinterpret_cast<float*>(b + F.sy_off);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_rmsnorm_rows(hidden, gamma, T, d, eps, y, status, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (launch_quantize_rows_e4m3(y, rows_padded(T), d, y8, sy, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (launch_lmhead_lse_fp8(y8, sy, W_codes, W_scales, token_ids, T, d, V, temperature, part, tgt,
                            status, st, sms) != cudaSuccess)
    return TIM_ERR_CUDA;
  return from_cuda(launch_lse_finalize(part, tgt, token_ids, T, V, out_logprob, out_lse, out_top1,
                                       status, st));
}

tim_status tim_split_tf32(const float* x, int64_t n, float* big, float* small,
                          tim_stream_t stream) {
  if (x == nullptr || big == nullptr || small == nullptr) return TIM_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(big, 16) || !aligned(small, 16)) return TIM_ERR_INVALID_ARG;
  if (n < 4 || (n % 4) != 0) return TIM_ERR_SHAPE;
  int sms = 0;
  tim_status s = check_device(&sms);
  if (s != TIM_OK) return s;
  return from_cuda(launch_split_tf32(x, n, big, small, reinterpret_cast<cudaStream_t>(stream), sms));
}

size_t tim_logprob_fp32_workspace_size(int64_t T, int32_t d, int32_t V) {
  if (check_shape(T, d, V) != TIM_OK) return 0;
  return fp32_layout(T, d, V).total;
}

tim_status tim_logprob_fp32(const void* hidden, const void* gamma, const float* W_big,
                            const float* W_small, const int32_t* token_ids, int64_t T, int32_t d,
                            int32_t V, float temperature, float eps, float* out_logprob,
                            float* out_lse, int32_t* out_top1, void* workspace,
                            size_t workspace_bytes, tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || W_big == nullptr || W_small == nullptr ||
      token_ids == nullptr || out_logprob == nullptr || out_lse == nullptr ||
      out_top1 == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16) || !aligned(W_big, 16) ||
      !aligned(W_small, 16) || !aligned(token_ids, 4) || !aligned(out_logprob, 4) ||
      !aligned(out_lse, 4) || !aligned(out_top1, 4))
    return TIM_ERR_INVALID_ARG;
  tim_status s = check_shape(T, d, V);
  if (s != TIM_OK) return s;
  if ((s = check_scalars(temperature, eps)) != TIM_OK) return s;
  const Fp32Layout F = fp32_layout(T, d, V);
  if ((s = check_workspace(workspace, workspace_bytes, F.total)) != TIM_OK) return s;
  int sms = 0;
  if ((s = check_device(&sms)) != TIM_OK) return s;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(b + F.base.status_off);
  void* part = b + F.base.part_off;
  float* tgt = reinterpret_cast<float*>(b + F.base.tgt_off);
  float* ybig = reinterpret_cast<float*>(b + F.ybig_off);
  float* ysmall = reinterpret_cast<float*>(b + F.ysmall_off);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_rmsnorm_rows_split(hidden, gamma, T, d, eps, ybig, ysmall, status, st) !=
      cudaSuccess)
    return TIM_ERR_CUDA;
  if (launch_lmhead_lse_tf32x3(ybig, ysmall, W_big, W_small, token_ids, T, d, V, temperature,
                               part, tgt, status, st, sms) != cudaSuccess)
    return TIM_ERR_CUDA;
  return from_cuda(launch_lse_finalize(part, tgt, token_ids, T, V, out_logprob, out_lse, out_top1,
                                       status, st));
}

size_t tim_logprob_backward_workspace_size(int64_t T, int32_t d, int32_t V) {
  if (check_shape(T, d, V) != TIM_OK) return 0;
  if (rows_padded(T) / 64 > 65535 || (static_cast<int64_t>(V) + 63) / 64 > 65535) return 0;
  return backward_layout(T, d, V).total;
}

tim_status tim_logprob_backward(const void* hidden, const void* gamma, const void* W,
                                const int32_t* token_ids, const float* lse,
                                const float* grad_logprob, int64_t T, int32_t d, int32_t V,
                                float temperature, float eps, float* out_dy, float* out_dW,
                                int32_t accumulate_dW, void* workspace, size_t workspace_bytes,
                                tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || W == nullptr || token_ids == nullptr ||
      lse == nullptr || grad_logprob == nullptr || out_dy == nullptr || out_dW == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16) || !aligned(W, 16) || !aligned(token_ids, 4) ||
      !aligned(lse, 4) || !aligned(grad_logprob, 4) || !aligned(out_dy, 16) ||
      !aligned(out_dW, 16))
    return TIM_ERR_INVALID_ARG;
  if (accumulate_dW != 0 && accumulate_dW != 1) return TIM_ERR_INVALID_ARG;
  tim_status s = check_shape(T, d, V);
  if (s != TIM_OK) return s;
  if ((s = check_scalars(temperature, eps)) != TIM_OK) return s;
  if (rows_padded(T) / 64 > 65535 || (static_cast<int64_t>(V) + 63) / 64 > 65535)
    return TIM_ERR_SHAPE;
  const BwdLayout B = backward_layout(T, d, V);
  if ((s = check_workspace(workspace, workspace_bytes, B.total)) != TIM_OK) return s;
  int sms = 0;
  if ((s = check_device(&sms)) != TIM_OK) return s;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(b + B.status_off);
  uint16_t* y = reinterpret_cast<uint16_t*>(b + B.y_off);
  uint16_t* gz = reinterpret_cast<uint16_t*>(b + B.g_off);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // y exactly as the forward computes it (same kernel)
  if (launch_rmsnorm_rows(hidden, gamma, T, d, eps, y, status, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  // G = dL/dz from the recomputed logits, row-major [Tp][Vp]
  if (launch_logit_grad(y, W, token_ids, lse, grad_logprob, T, d, V, temperature, gz, B.Vp,
                        status, st, sms) != cudaSuccess)
    return TIM_ERR_CUDA;
  // dL/dy = G . W: A = G K-major [Tp][Vp] (K = V), B = W read MN-major ([V][d], d contiguous)
  if (launch_gemm_store(gz, B.Tp, B.Vp, 0, W, d, d, 1, V, T, out_dy, d, 0, status, st, sms) !=
      cudaSuccess)
    return TIM_ERR_CUDA;
  // dL/dW = G^T . y: A = G read MN-major ([T][Vp], V contiguous; K = T), B = y read
  // MN-major ([T][d], d contiguous)
  return from_cuda(launch_gemm_store(gz, V, B.Vp, 1, y, d, d, 1, T, V, out_dW, d, accumulate_dW,
                                     status, st, sms));
}

// Self-test shapes: one 128-row tile group against two vocabulary tiles.
constexpr int64_t kSelftestT = 128;
constexpr int32_t kSelftestD = 64;
constexpr int32_t kSelftestV = 512;

size_t tim_selftest_workspace_size(void) {
  const size_t base = logprob_layout(kSelftestT, kSelftestD, kSelftestV).total;
  return align_up(base + static_cast<size_t>(kSelftestV) * kSelftestD * 2, 1024) +
         align_up(static_cast<size_t>(kSelftestT) * 4, 1024);
}

tim_status tim_selftest_wait_timeout(int32_t limit_ms, void* workspace, size_t workspace_bytes,
                                     tim_stream_t stream) {
  if (limit_ms < 1 || limit_ms > 2000) return TIM_ERR_INVALID_ARG;
  tim_status s = check_workspace(workspace, workspace_bytes, tim_selftest_workspace_size());
  if (s != TIM_OK) return s;
  int sms = 0;
  if ((s = check_device(&sms)) != TIM_OK) return s;
  const WsLayout L = logprob_layout(kSelftestT, kSelftestD, kSelftestV);
  uint8_t* b = static_cast<uint8_t*>(workspace);
  const size_t w_off = align_up(L.total, 1024);
  const size_t ids_off = align_up(w_off + static_cast<size_t>(kSelftestV) * kSelftestD * 2, 1024);
  return from_cuda(launch_wait_selftest(
      b + L.y_off, b + w_off, reinterpret_cast<const int32_t*>(b + ids_off), kSelftestT,
      kSelftestD, kSelftestV, b + L.part_off, reinterpret_cast<float*>(b + L.tgt_off),
      reinterpret_cast<int*>(b + L.status_off),
      static_cast<uint64_t>(limit_ms) * 1000ull * 1000ull, reinterpret_cast<cudaStream_t>(stream),
      sms));
}

// RMSNorm-backward workspace: status | rstd [T] | dgamma partials [chunks][d].
size_t tim_rmsnorm_backward_workspace_size(int64_t T, int32_t d) {
  if (T < 1 || T > INT32_MAX || d < 64 || d > 65536 || (d % 64) != 0 ||
      rmsnorm_backward_chunks(T) > 65535)
    return 0;
  return align_up(1024 + static_cast<size_t>(T) * 4, 1024) +
         align_up(static_cast<size_t>(rmsnorm_backward_chunks(T)) * d * 4, 1024);
}

tim_status tim_rmsnorm_backward(const void* hidden, const void* gamma, const float* dy, int64_t T,
                                int32_t d, float eps, float* out_dh, float* out_dgamma,
                                int32_t accumulate_dgamma, void* workspace,
                                size_t workspace_bytes, tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || dy == nullptr || out_dh == nullptr ||
      out_dgamma == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16) || !aligned(dy, 16) || !aligned(out_dh, 16) ||
      !aligned(out_dgamma, 4))
    return TIM_ERR_INVALID_ARG;
  if (accumulate_dgamma != 0 && accumulate_dgamma != 1) return TIM_ERR_INVALID_ARG;
  if (T < 1 || T > INT32_MAX || d < 64 || d > 65536 || (d % 64) != 0 ||
      rmsnorm_backward_chunks(T) > 65535)
    return TIM_ERR_SHAPE;
  if (!(std::isfinite(eps) && eps >= 0.f)) return TIM_ERR_INVALID_ARG;
  tim_status s =
      check_workspace(workspace, workspace_bytes, tim_rmsnorm_backward_workspace_size(T, d));
  if (s != TIM_OK) return s;
  if ((s = check_device(nullptr)) != TIM_OK) return s;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  float* rstd = reinterpret_cast<float*>(b + 1024);
  float* partial = reinterpret_cast<float*>(b + align_up(1024 + static_cast<size_t>(T) * 4, 1024));
  return from_cuda(launch_rmsnorm_backward(hidden, gamma, dy, T, d, eps, out_dh, out_dgamma,
                                           accumulate_dgamma, rstd, partial,
                                           reinterpret_cast<int*>(b),
                                           reinterpret_cast<cudaStream_t>(stream)));
}

size_t tim_processed_logprob_workspace_size(int64_t T, int32_t d, int32_t V) {
  if (check_shape(T, d, V) != TIM_OK) return 0;
  return processed_layout(T, d, V).total;
}

tim_status tim_processed_logprob(const void* hidden, const void* gamma, const void* W,
                                 const int32_t* token_ids, int64_t T, int32_t d, int32_t V,
                                 float temperature, float eps, int32_t top_k, float top_p,
                                 float* out_logprob, float* out_lse_kept, int32_t* out_kept,
                                 void* workspace, size_t workspace_bytes, tim_stream_t stream) {
  return tim_processed_logprob_head(hidden, gamma, W, token_ids, T, d, V, temperature, eps, top_k,
                                    top_p, out_logprob, out_lse_kept, out_kept, nullptr, nullptr,
                                    workspace, workspace_bytes, stream);
}

tim_status tim_processed_logprob_head(const void* hidden, const void* gamma, const void* W,
                                      const int32_t* token_ids, int64_t T, int32_t d, int32_t V,
                                      float temperature, float eps, int32_t top_k, float top_p,
                                      float* out_logprob, float* out_lse_kept, int32_t* out_kept,
                                      int32_t* out_head_ids, float* out_head_logprob,
                                      void* workspace, size_t workspace_bytes,
                                      tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || W == nullptr || token_ids == nullptr ||
      out_logprob == nullptr || out_lse_kept == nullptr || out_kept == nullptr)
    return TIM_ERR_INVALID_ARG;
  if ((out_head_ids == nullptr) != (out_head_logprob == nullptr)) return TIM_ERR_INVALID_ARG;
  if (out_head_ids != nullptr && (!aligned(out_head_ids, 4) || !aligned(out_head_logprob, 4)))
    return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16) || !aligned(W, 16) || !aligned(token_ids, 4) ||
      !aligned(out_logprob, 4) || !aligned(out_lse_kept, 4) || !aligned(out_kept, 4))
    return TIM_ERR_INVALID_ARG;
  tim_status s = check_shape(T, d, V);
  if (s != TIM_OK) return s;
  if ((s = check_scalars(temperature, eps)) != TIM_OK) return s;
  if (top_k < 1 || top_k > TIM_PROCESSED_MAX_K) return TIM_ERR_INVALID_ARG;
  if (!(std::isfinite(top_p) && top_p > 0.f && top_p <= 1.f)) return TIM_ERR_INVALID_ARG;
  const int n_tiles = (V + kBN - 1) / kBN;
  if (n_tiles > TIM_PROCESSED_CAPACITY) return TIM_ERR_SHAPE;
  if (n_tiles < top_k && V > TIM_PROCESSED_CAPACITY) return TIM_ERR_SHAPE;
  const ProcLayout P = processed_layout(T, d, V);
  if ((s = check_workspace(workspace, workspace_bytes, P.total)) != TIM_OK) return s;
  int sms = 0;
  if ((s = check_device(&sms)) != TIM_OK) return s;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(b + P.base.status_off);
  void* y = b + P.base.y_off;
  float* thr = reinterpret_cast<float*>(b + P.thr_off);
  int* cnt = reinterpret_cast<int*>(b + P.cnt_off);
  void* cand = b + P.cand_off;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_rmsnorm_rows(hidden, gamma, T, d, eps, y, status, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  void* top4 = b + P.top4_off;
  int* fb_n = reinterpret_cast<int*>(b + P.fbn_off);
  int* fb_rows = reinterpret_cast<int*>(b + P.fbrows_off);
  void* y_fb = b + P.yfb_off;
  if (launch_lmhead_top4(y, W, token_ids, T, d, V, top4, status, st, sms) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (cudaMemsetAsync(fb_n, 0, sizeof(int), st) != cudaSuccess) return TIM_ERR_CUDA;
  if (launch_topk_candidates(top4, T, V, top_k, thr, cnt, cand, TIM_PROCESSED_CAPACITY, fb_n,
                             fb_rows, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  // rows whose candidates the top-4 lists cannot vouch for: gathered and rescored
  if (launch_gather_rows(y, fb_rows, fb_n, T, d, y_fb, st, sms) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (launch_lmhead_collect(y_fb, W, token_ids, T, d, V, temperature, thr, cnt, cand,
                            TIM_PROCESSED_CAPACITY, fb_n, fb_rows, status, st, sms) !=
      cudaSuccess)
    return TIM_ERR_CUDA;
  return from_cuda(launch_topk_finalize(cand, cnt, token_ids, T, V, top_k, top_p, temperature,
                                        TIM_PROCESSED_CAPACITY, out_logprob, out_lse_kept,
                                        out_kept, out_head_ids, out_head_logprob, status, st));
}

tim_status tim_vocab_shard(int32_t V, int32_t G, int32_t g, int32_t* v0, int32_t* v_len) {
  if (v0 == nullptr || v_len == nullptr || !valid_shard(G, g)) return TIM_ERR_INVALID_ARG;
  if (V < 1 || V > INT32_MAX - 256) return TIM_ERR_SHAPE;
  int a = 0, n = 0;
  vocab_shard_range(V, G, g, &a, &n);
  *v0 = a;
  *v_len = n;
  return TIM_OK;
}

size_t tim_logprob_shard_workspace_size(int64_t T, int32_t d, int32_t V, int32_t G, int32_t g) {
  if (check_shape(T, d, V) != TIM_OK || !valid_shard(G, g)) return 0;
  int v0 = 0, v_len = 0;
  vocab_shard_range(V, G, g, &v0, &v_len);
  return logprob_layout(T, d, v_len > 0 ? v_len : 1).total;
}

tim_status tim_logprob_shard(const void* hidden, const void* gamma, const void* W_shard,
                             const int32_t* token_ids, int64_t T, int32_t d, int32_t V,
                             int32_t G, int32_t g, float temperature, float eps, void* out_rec,
                             float* out_tgt, void* workspace, size_t workspace_bytes,
                             tim_stream_t stream) {
  if (hidden == nullptr || gamma == nullptr || token_ids == nullptr || out_rec == nullptr ||
      out_tgt == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!valid_shard(G, g)) return TIM_ERR_INVALID_ARG;
  tim_status s = check_shape(T, d, V);
  if (s != TIM_OK) return s;
  if ((s = check_scalars(temperature, eps)) != TIM_OK) return s;
  int v0 = 0, v_len = 0;
  vocab_shard_range(V, G, g, &v0, &v_len);
  if (v_len > 0 && W_shard == nullptr) return TIM_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(gamma, 16) || (W_shard != nullptr && !aligned(W_shard, 16)) ||
      !aligned(token_ids, 4) || !aligned(out_rec, 16) || !aligned(out_tgt, 4))
    return TIM_ERR_INVALID_ARG;
  if ((s = check_workspace(workspace, workspace_bytes,
                           tim_logprob_shard_workspace_size(T, d, V, G, g))) != TIM_OK)
    return s;
  int sms = 0;
  if ((s = check_device(&sms)) != TIM_OK) return s;
  if (v_len == 0) return TIM_OK;  // this rank owns no vocabulary: its records are never read
  const Ptrs p = logprob_ptrs(workspace, T, d, v_len);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (launch_rmsnorm_rows(hidden, gamma, T, d, eps, p.y, p.status, st) != cudaSuccess)
    return TIM_ERR_CUDA;
  if (launch_lmhead_lse_shard(p.y, W_shard, token_ids, T, d, v_len, v0, temperature, p.part,
                              p.tgt, p.status, st, sms) != cudaSuccess)
    return TIM_ERR_CUDA;
  return from_cuda(launch_shard_reduce(p.part, p.tgt, T, V, G, g, v_len, out_rec, out_tgt, st));
}

size_t tim_logprob_merge_workspace_size(int64_t T) { return T < 1 ? 0 : 1024; }

tim_status tim_logprob_merge_shards(const void* recs, const float* tgts, const int32_t* token_ids,
                                    int64_t T, int32_t V, int32_t G, float* out_logprob,
                                    float* out_lse, int32_t* out_top1, void* workspace,
                                    size_t workspace_bytes, tim_stream_t stream) {
  if (recs == nullptr || tgts == nullptr || token_ids == nullptr || out_logprob == nullptr ||
      out_lse == nullptr || out_top1 == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!valid_shard(G, 0)) return TIM_ERR_INVALID_ARG;
  if (!aligned(recs, 16) || !aligned(tgts, 4) || !aligned(token_ids, 4) ||
      !aligned(out_logprob, 4) || !aligned(out_lse, 4) || !aligned(out_top1, 4))
    return TIM_ERR_INVALID_ARG;
  if (T < 1 || T > INT32_MAX || V < 1 || V > INT32_MAX - 256) return TIM_ERR_SHAPE;
  tim_status s = check_workspace(workspace, workspace_bytes, tim_logprob_merge_workspace_size(T));
  if (s != TIM_OK) return s;
  if ((s = check_device(nullptr)) != TIM_OK) return s;
  return from_cuda(launch_merge_shards(recs, tgts, token_ids, T, V, G, out_logprob, out_lse,
                                       out_top1, static_cast<int*>(workspace),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

size_t tim_compare_diag_workspace_size(int64_t T, int32_t n_seq) {
  if (T < 1 || n_seq < 1) return 0;
  return diag_workspace_bytes(T, n_seq);
}

tim_status tim_compare_diag(const float* lp_gen, const float* lp_replay, const float* lp_train,
                            const int32_t* top1_gen, const int32_t* top1_replay,
                            const int32_t* top1_train, const int64_t* seq_offsets, int32_t n_seq,
                            const uint8_t* mask, int64_t T, float tis_cap, float mis_lo,
                            float mis_hi, tim_seq_diag* out_diag, void* workspace,
                            size_t workspace_bytes, tim_stream_t stream) {
  if (lp_gen == nullptr || lp_replay == nullptr || lp_train == nullptr || seq_offsets == nullptr ||
      mask == nullptr || out_diag == nullptr)
    return TIM_ERR_INVALID_ARG;
  if (!aligned(lp_gen, 4) || !aligned(lp_replay, 4) || !aligned(lp_train, 4) ||
      !aligned(seq_offsets, 8) || !aligned(out_diag, 8) ||
      (top1_gen != nullptr && !aligned(top1_gen, 4)) ||
      (top1_replay != nullptr && !aligned(top1_replay, 4)) ||
      (top1_train != nullptr && !aligned(top1_train, 4)))
    return TIM_ERR_INVALID_ARG;
  if (T < 1 || T > INT32_MAX || n_seq < 1) return TIM_ERR_SHAPE;
  if (!(std::isfinite(tis_cap) && tis_cap > 0.f)) return TIM_ERR_INVALID_ARG;
  if (!(std::isfinite(mis_lo) && std::isfinite(mis_hi) && mis_lo > 0.f && mis_lo <= mis_hi))
    return TIM_ERR_INVALID_ARG;
  tim_status s =
      check_workspace(workspace, workspace_bytes, tim_compare_diag_workspace_size(T, n_seq));
  if (s != TIM_OK) return s;
  if ((s = check_device(nullptr)) != TIM_OK) return s;
  return from_cuda(launch_seg_diag(lp_gen, lp_replay, lp_train, top1_gen, top1_replay, top1_train,
                                   seq_offsets, n_seq, mask, T, tis_cap, mis_lo, mis_hi, out_diag,
                                   workspace, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
