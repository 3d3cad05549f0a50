// qat_api.cu -- the C ABI declared in include/qat_attn.h: host-side validation, the
// backward workspace layout, kernel launches on the caller's stream, status codes and
// the device-side error word.  No entry point here allocates device memory.
#include "qat_attn.h"
#include "qat_internal.h"
#include "sm100.cuh"

#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

namespace qat {

// The error word that kernels whose bounded waits expire set (read and cleared by
// qat_attn_device_status), followed by the limit of those waits.
__device__ sm100::DeviceState g_device_state = {0u, 0u, sm100::kWaitLimitNs};

cudaError_t read_and_clear_device_error(unsigned int* out, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_device_state, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0u;
  return cudaMemcpyToSymbol(g_device_state, &zero, sizeof(unsigned int));
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_ctx_mu;
int g_num_sms[kMaxDevices] = {};
}  // namespace

cudaError_t device_context(unsigned int** err, int* num_sms) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // a host-side lookup (no allocation), repeated on every call: a cached address would
  // go stale when the device's context is destroyed and recreated
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_device_state);
  if (e != cudaSuccess) return e;
  *err = static_cast<unsigned int*>(p);
  std::lock_guard<std::mutex> lock(g_ctx_mu);
  if (g_num_sms[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = n;
  }
  *num_sms = g_num_sms[dev];
  return cudaSuccess;
}

}  // namespace qat

namespace {

using qat::aligned16;
using qat::check_sizes;
using qat::kMaxRows;

constexpr float kLog2e = 1.4426950408889634f;
constexpr size_t kAlign = 256;

// With QAT_VERBOSE=1 in the environment, CUDA errors are also printed to stderr.
qat_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return QAT_OK;
  static const bool verbose = [] {
    const char* v = getenv("QAT_VERBOSE");
    return v != nullptr && v[0] == '1';
  }();
  if (verbose) fprintf(stderr, "qat_attn: CUDA error %d: %s\n", static_cast<int>(e), cudaGetErrorString(e));
  return QAT_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* qat_status_string(qat_status_t status) {
  switch (status) {
    case QAT_OK: return "QAT_OK";
    case QAT_ERR_INVALID_ARG: return "QAT_ERR_INVALID_ARG: invalid argument";
    case QAT_ERR_UNSUPPORTED: return "QAT_ERR_UNSUPPORTED: unsupported configuration";
    case QAT_ERR_CUDA: return "QAT_ERR_CUDA: CUDA runtime or launch error";
    case QAT_ERR_TIMEOUT: return "QAT_ERR_TIMEOUT: a bounded device wait expired";
    case QAT_ERR_WORKSPACE: return "QAT_ERR_WORKSPACE: workspace missing or too small";
  }
  return "QAT_ERR_UNKNOWN: unknown status code";
}

qat_status_t qat_attn_fwd(const void* q, const void* k, const void* v, void* o_q, void* o_hp,
                          float* lse, int B, int H, int Nq, int Nkv, int D, float sm_scale,
                          int causal, int quant_mode, void* stream) {
  bool empty = false;
  const qat_status_t st = check_sizes(B, H, Nq, Nkv, D, sm_scale, causal, quant_mode, &empty);
  if (st != QAT_OK || empty) return st;
  const void* ptrs[] = {q, k, v, o_q, o_hp, lse};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return QAT_ERR_INVALID_ARG;
  qat::FwdArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.o_q = static_cast<uint16_t*>(o_q);
  a.o_hp = static_cast<uint16_t*>(o_hp);
  a.lse = lse;
  a.B = B; a.H = H; a.Nq = Nq; a.Nkv = Nkv; a.D = D;
  a.sm_scale = sm_scale;
  a.qk_scale = sm_scale * kLog2e;
  a.causal = causal;
  a.quant = quant_mode != QAT_QUANT_NONE;
  a.kv_head_rows = Nkv;
  a.o_q_f32 = nullptr;
  a.o_hp_f32 = nullptr;
  unsigned int* err = nullptr;
  int num_sms = 0;
  cudaError_t e = qat::device_context(&err, &num_sms);
  if (e == cudaSuccess) e = qat::launch_fwd_tc(a, err, num_sms, static_cast<cudaStream_t>(stream));
  return from_cuda(e);
}

qat_status_t qat_attn_fwd_chunk(const void* q, const void* k, const void* v, float* o_q,
                                float* o_hp, float* lse, int B, int H, int Nq, int Nkv_total,
                                int kv_begin, int kv_len, int D, float sm_scale, int quant_mode,
                                void* stream) {
  bool empty = false;
  const qat_status_t st = check_sizes(B, H, Nq, Nkv_total, D, sm_scale, 0, quant_mode, &empty);
  if (st != QAT_OK || empty) return st;
  if (kv_begin < 0 || kv_len < 1 || static_cast<long long>(kv_begin) + kv_len > Nkv_total)
    return QAT_ERR_INVALID_ARG;
  if (kv_begin % 64 != 0) return QAT_ERR_UNSUPPORTED;  // a quantization tile would be split
  const void* ptrs[] = {q, k, v, o_q, o_hp, lse};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return QAT_ERR_INVALID_ARG;
  const size_t off = static_cast<size_t>(kv_begin) * D;
  qat::FwdArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k) + off;
  a.v = static_cast<const uint16_t*>(v) + off;
  a.o_q = nullptr;
  a.o_hp = nullptr;
  a.lse = lse;
  a.B = B; a.H = H; a.Nq = Nq; a.Nkv = kv_len; a.D = D;
  a.sm_scale = sm_scale;
  a.qk_scale = sm_scale * kLog2e;
  a.causal = 0;
  a.quant = quant_mode != QAT_QUANT_NONE;
  a.kv_head_rows = Nkv_total;
  a.o_q_f32 = o_q;
  a.o_hp_f32 = o_hp;
  unsigned int* err = nullptr;
  int num_sms = 0;
  cudaError_t e = qat::device_context(&err, &num_sms);
  if (e == cudaSuccess) e = qat::launch_fwd_tc(a, err, num_sms, static_cast<cudaStream_t>(stream));
  return from_cuda(e);
}

qat_status_t qat_attn_merge(float* o_q_acc, float* o_hp_acc, float* lse_acc,
                            const float* o_q_part, const float* o_hp_part, const float* lse_part,
                            void* o_q_out, void* o_hp_out, int B, int H, int Nq, int D,
                            void* stream) {
  if (B < 0 || H < 0 || Nq < 0 || (D != 64 && D != 128)) return QAT_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * Nq;
  if (rows > kMaxRows) return QAT_ERR_INVALID_ARG;
  if (rows == 0) return QAT_OK;
  const void* ptrs[] = {o_q_acc, o_hp_acc, lse_acc, o_q_part, o_hp_part, lse_part};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return QAT_ERR_INVALID_ARG;
  if ((o_q_out != nullptr && !aligned16(o_q_out)) || (o_hp_out != nullptr && !aligned16(o_hp_out)))
    return QAT_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int num_sms = 0;
  cudaError_t e = qat::device_context(&err, &num_sms);
  if (e == cudaSuccess)
    e = qat::launch_merge(o_q_acc, o_hp_acc, lse_acc, o_q_part, o_hp_part, lse_part,
                          static_cast<uint16_t*>(o_q_out), static_cast<uint16_t*>(o_hp_out), rows,
                          D, num_sms, static_cast<cudaStream_t>(stream));
  return from_cuda(e);
}

size_t qat_attn_bwd_workspace_bytes(int B, int H, int Nq, int Nkv, int D) {
  bool empty = false;
  if (check_sizes(B, H, Nq, Nkv, D, 1.0f, 0, 0, &empty) != QAT_OK) return 0;
  return qat::bwd_workspace_layout(B, H, Nq, Nkv, D, qat::bwd_stream_k_ctas(B, H, Nq, Nkv)).total;
}

}  // extern "C"

namespace {

qat_status_t bwd_impl(const void* q, const void* k, const void* v, const void* o_hp,
                      const float* lse, const void* dO, void* dq, void* dk, void* dv,
                      const float* k_mean, int B, int H, int Nq, int Nkv, int D, float sm_scale,
                      int causal, int quant_mode, void* workspace, size_t workspace_bytes,
                      void* stream) {
  bool empty = false;
  const qat_status_t st = check_sizes(B, H, Nq, Nkv, D, sm_scale, causal, quant_mode, &empty);
  if (st != QAT_OK) return st;
  if (B == 0 || H == 0) return QAT_OK;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t kv_bytes = static_cast<size_t>(B) * H * Nkv * D * sizeof(uint16_t);
  if (Nq == 0) {  // no queries: every key gets zero gradient
    if (dk == nullptr || dv == nullptr || !aligned16(dk) || !aligned16(dv))
      return QAT_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(dk, 0, kv_bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_bytes, s);
    return from_cuda(e);
  }
  const void* ptrs[] = {q, k, v, o_hp, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return QAT_ERR_INVALID_ARG;
  // the stream-K split of the dK/dV work runs only when the workspace also holds its
  // segment sums (qat_attn_bwd_workspace_bytes does; the no-alloc scratch may not)
  const size_t need = qat::bwd_workspace_layout(B, H, Nq, Nkv, D, 0).total;
  if (workspace == nullptr || workspace_bytes < need) return QAT_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return QAT_ERR_INVALID_ARG;
  int sk = causal ? 0 : qat::bwd_stream_k_ctas(B, H, Nq, Nkv);
  if (sk > 0 && workspace_bytes < qat::bwd_workspace_layout(B, H, Nq, Nkv, D, sk).total) sk = 0;

  qat::BwdArgs a;
  const qat::BwdWorkspace wl = qat::bwd_workspace_layout(B, H, Nq, Nkv, D, sk);
  char* ws = static_cast<char*>(workspace);
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.o_hp = static_cast<const uint16_t*>(o_hp);
  a.lse = lse;
  a.dO = static_cast<const uint16_t*>(dO);
  a.dq = static_cast<uint16_t*>(dq);
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.lse_pad = reinterpret_cast<float*>(ws + wl.off_lse);
  a.delta = reinterpret_cast<float*>(ws + wl.off_delta);
  a.lse_ext = reinterpret_cast<uint16_t*>(ws + wl.off_lse_ext);
  a.d_ext = reinterpret_cast<uint16_t*>(ws + wl.off_d_ext);
  a.ones = reinterpret_cast<uint16_t*>(ws + wl.off_ones);
  a.part = sk > 0 ? reinterpret_cast<float*>(ws + wl.off_part) : nullptr;
  a.k_mean = k_mean;
  a.sk_ctas = sk;
  a.B = B; a.H = H; a.Nq = Nq; a.Nkv = Nkv; a.D = D;
  a.sm_scale = sm_scale;
  a.qk_scale = sm_scale * kLog2e;
  a.causal = causal;
  a.page_bwd = quant_mode == QAT_QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD;
  unsigned int* err = nullptr;
  int num_sms = 0;
  cudaError_t e = qat::device_context(&err, &num_sms);
  if (e == cudaSuccess) e = qat::launch_bwd_tc(a, err, num_sms, s);
  return from_cuda(e);
}

}  // namespace

extern "C" {

qat_status_t qat_attn_bwd(const void* q, const void* k, const void* v, const void* o_hp,
                          const float* lse, const void* dO, void* dq, void* dk, void* dv,
                          int B, int H, int Nq, int Nkv, int D, float sm_scale, int causal,
                          int quant_mode, void* workspace, size_t workspace_bytes,
                          void* stream) {
  return bwd_impl(q, k, v, o_hp, lse, dO, dq, dk, dv, nullptr, B, H, Nq, Nkv, D, sm_scale,
                  causal, quant_mode, workspace, workspace_bytes, stream);
}

qat_status_t qat_attn_bwd_smooth_k(const void* q, const void* k, const void* v,
                                   const void* o_hp, const float* lse, const void* dO, void* dq,
                                   void* dk, void* dv, const float* k_mean, int B, int H, int Nq,
                                   int Nkv, int D, float sm_scale, int causal, int quant_mode,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (k_mean == nullptr || !aligned16(k_mean)) return QAT_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o_hp, lse, dO, dq, dk, dv, k_mean, B, H, Nq, Nkv, D, sm_scale,
                  causal, quant_mode, workspace, workspace_bytes, stream);
}

qat_status_t qat_debug_set_wait_limit_us(int limit_us, void* stream) {
  if (limit_us < 0 || limit_us > 4000000) return QAT_ERR_INVALID_ARG;
  // no kernel of the library may be running while the limit changes
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  const unsigned long long ns =
      limit_us == 0 ? 1ull : static_cast<unsigned long long>(limit_us) * 1000ull;
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbol(qat::g_device_state, &ns, sizeof(ns),
                           offsetof(qat::sm100::DeviceState, wait_limit_ns));
  return from_cuda(e);
}

qat_status_t qat_attn_device_status(void* stream) {
  unsigned int word = 0u;
  const cudaError_t e = qat::read_and_clear_device_error(&word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return QAT_ERR_CUDA;
  return word ? QAT_ERR_TIMEOUT : QAT_OK;
}

qat_status_t qat_channel_mean(const void* x, float* mean, int B, int H, int N, int D,
                              void* stream) {
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128)) return QAT_ERR_INVALID_ARG;
  if (mean == nullptr || (reinterpret_cast<uintptr_t>(mean) & 3u) != 0) return QAT_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows > kMaxRows) return QAT_ERR_INVALID_ARG;
  if (rows > 0 && (x == nullptr || !aligned16(x))) return QAT_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int num_sms = 0;
  cudaError_t e = qat::device_context(&err, &num_sms);
  if (e == cudaSuccess)
    e = qat::launch_channel_mean(static_cast<const uint16_t*>(x), mean, rows, D, num_sms,
                                 static_cast<cudaStream_t>(stream));
  return from_cuda(e);
}

qat_status_t qat_fake_quant_tokens(const void* x, const float* mean, void* out, float* scales,
                                   int B, int H, int N, int D, void* stream) {
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128)) return QAT_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh * N > kMaxRows || bh * ((N + 31) / 32) > kMaxRows) return QAT_ERR_INVALID_ARG;
  if (bh * N == 0) return QAT_OK;
  if (x == nullptr || out == nullptr || !aligned16(x) || !aligned16(out)) return QAT_ERR_INVALID_ARG;
  if (mean != nullptr && (reinterpret_cast<uintptr_t>(mean) & 3u) != 0) return QAT_ERR_INVALID_ARG;
  if (scales != nullptr && (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return QAT_ERR_INVALID_ARG;
  return from_cuda(qat::launch_fake_quant_tokens(
      static_cast<const uint16_t*>(x), mean, static_cast<uint16_t*>(out), scales,
      static_cast<int>(bh), N, D, static_cast<cudaStream_t>(stream)));
}

qat_status_t qat_subtract_mean(const void* x, const float* mean, void* out, int B, int H, int N,
                               int D, void* stream) {
  if (B < 0 || H < 0 || N < 0 || (D != 64 && D != 128)) return QAT_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows > kMaxRows) return QAT_ERR_INVALID_ARG;
  if (rows == 0) return QAT_OK;
  if (x == nullptr || out == nullptr || mean == nullptr || !aligned16(x) || !aligned16(out) ||
      !aligned16(mean))
    return QAT_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int num_sms = 0;
  cudaError_t e = qat::device_context(&err, &num_sms);
  if (e == cudaSuccess)
    e = qat::launch_subtract_mean(static_cast<const uint16_t*>(x), mean,
                                  static_cast<uint16_t*>(out), rows, D, num_sms,
                                  static_cast<cudaStream_t>(stream));
  return from_cuda(e);
}

qat_status_t qat_debug_quant_tiles(const float* p, int rows, int cols, float* deq, float* scales,
                                   unsigned char* codes, void* stream) {
  if (rows < 0 || cols < 0) return QAT_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return QAT_OK;
  if (p == nullptr || deq == nullptr || scales == nullptr || codes == nullptr)
    return QAT_ERR_INVALID_ARG;
  return from_cuda(qat::launch_debug_quant(p, rows, cols, deq, scales, codes,
                                           static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
