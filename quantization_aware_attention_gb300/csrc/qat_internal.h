// qat_internal.h -- declarations shared by the library's translation units (not ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qat {

// Arguments of one forward launch (device pointers, validated by the ABI layer).
struct FwdArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  uint16_t* o_q;
  uint16_t* o_hp;
  float* lse;
  int B, H, Nq, Nkv, D;
  float sm_scale;
  float qk_scale;  // sm_scale * log2(e)
  int causal;
  int quant;
};

// Arguments of one backward launch.
struct BwdArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const uint16_t* o_hp;
  const float* lse;
  const uint16_t* dO;
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  float* delta;     // fp32 [B, H, Nq] in the workspace
  int B, H, Nq, Nkv, D;
  float sm_scale;
  float qk_scale;
  int causal;
};

// Kernel launchers (return cudaGetLastError() after the launches).
cudaError_t launch_fwd_tc(const FwdArgs& a, unsigned int* err, int num_sms, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_mma(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_debug_quant(const float* p, int rows, int cols, float* deq,
                               float* scales, uint8_t* codes, cudaStream_t s);

// Device-side error word (bounded waits set it); defined in qat_api.cu.
cudaError_t read_and_clear_device_error(unsigned int* out, cudaStream_t s);
// Device address of that word and the SM count, for the current device (cached).
cudaError_t device_context(unsigned int** err, int* num_sms);

}  // namespace qat
