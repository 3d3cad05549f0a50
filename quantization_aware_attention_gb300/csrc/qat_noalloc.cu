// qat_noalloc.cu -- qat_attn_bwd_noalloc: the backward pass for callers that cannot
// provide device scratch memory.
//
// qat_attn_bwd asks its caller for a workspace.  Some callers cannot allocate one:
// a host program whose device memory is owned entirely by another runtime's pool (so it
// has no allocator it may call), or a process that must not allocate once it is
// running, because an allocation can block on the device or fail under memory pressure
// in the middle of a training step.  This entry point needs no workspace: its scratch
// is a fixed array compiled into this library, so every GPU that loads the library
// holds kNoAllocScratchBytes of device memory until the process exits.
//
// The array is shared by every call on a device and keeps the last call's contents.
// The backward overwrites every scratch value it reads (Delta is written in full by
// the preprocess kernel before the main kernels read it), so nothing needs clearing.
// Calls that overlap on the GPU (on different streams, or from different host
// threads without ordering) race on the array and give undefined results; order them.
#include "qat_attn.h"
#include "qat_internal.h"

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

// The scratch.  In host code this name is only a stand-in for the device symbol: its
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on the first
// call on each device, with that device current).
qat_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return QAT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QAT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return QAT_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QAT_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" qat_status_t qat_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                             const void* o_hp, const float* lse,
                                             const void* dO, void* dq, void* dk, void* dv,
                                             int B, int H, int Nq, int Nkv, int D,
                                             float sm_scale, int causal, int quant_mode,
                                             void* stream) {
  // Invalid sizes, or no query rows: qat_attn_bwd validates and needs no scratch.
  if (qat_attn_bwd_workspace_bytes(B, H, Nq, Nkv, D) == 0 || B == 0 || H == 0 || Nq == 0)
    return qat_attn_bwd(q, k, v, o_hp, lse, dO, dq, dk, dv, B, H, Nq, Nkv, D, sm_scale, causal,
                        quant_mode, nullptr, 0, stream);
  // the scratch must hold the workspace without the dK/dV query-part sums; qat_attn_bwd
  // uses the split only when those fit as well
  if (qat::bwd_workspace_layout(B, H, Nq, Nkv, D, 1).total > kNoAllocScratchBytes)
    return QAT_ERR_WORKSPACE;
  const void* ptrs[] = {q, k, v, o_hp, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return QAT_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const qat_status_t st = scratch_on_current_device(&scratch);
  if (st != QAT_OK) return st;
  return qat_attn_bwd(q, k, v, o_hp, lse, dO, dq, dk, dv, B, H, Nq, Nkv, D, sm_scale, causal,
                      quant_mode, scratch, kNoAllocScratchBytes, stream);
}
