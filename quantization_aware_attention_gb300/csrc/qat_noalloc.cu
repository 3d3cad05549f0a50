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

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

// The scratch.  In host code this name is only a stand-in for the device symbol: its
// device address comes from cudaGetSymbolAddress, with the device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  Looked up on every call (a
// host-side table lookup that allocates nothing): a cached address would go stale if the
// device's context were destroyed and recreated (cudaDeviceReset).  The first call on a
// device loads the library's device code there.
qat_status_t scratch_on_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return QAT_ERR_CUDA;
  *out = p;
  return QAT_OK;
}

}  // namespace

extern "C" qat_status_t qat_attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                             const void* o_hp, const float* lse,
                                             const void* dO, void* dq, void* dk, void* dv,
                                             int B, int H, int Nq, int Nkv, int D,
                                             float sm_scale, int causal, int quant_mode,
                                             void* stream) {
  // the same argument checks as qat_attn_bwd, in the same order, before the scratch size
  bool empty = false;
  const qat_status_t st = qat::check_sizes(B, H, Nq, Nkv, D, sm_scale, causal, quant_mode, &empty);
  if (st != QAT_OK) return st;
  // no query rows: qat_attn_bwd only zeroes dK and dV and needs no scratch
  if (empty)
    return qat_attn_bwd(q, k, v, o_hp, lse, dO, dq, dk, dv, B, H, Nq, Nkv, D, sm_scale, causal,
                        quant_mode, nullptr, 0, stream);
  const void* ptrs[] = {q, k, v, o_hp, lse, dO, dq, dk, dv};
  for (const void* p : ptrs)
    if (p == nullptr || !qat::aligned16(p)) return QAT_ERR_INVALID_ARG;
  // the scratch must hold the workspace without the dK/dV segment sums; qat_attn_bwd
  // uses the stream-K split only when those fit as well
  if (qat::bwd_workspace_layout(B, H, Nq, Nkv, D, 0).total > kNoAllocScratchBytes)
    return QAT_ERR_WORKSPACE;
  void* scratch = nullptr;
  const qat_status_t sst = scratch_on_current_device(&scratch);
  if (sst != QAT_OK) return sst;
  return qat_attn_bwd(q, k, v, o_hp, lse, dO, dq, dk, dv, B, H, Nq, Nkv, D, sm_scale, causal,
                      quant_mode, scratch, kNoAllocScratchBytes, stream);
}
