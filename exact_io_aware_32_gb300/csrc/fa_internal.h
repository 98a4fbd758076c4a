// Internal interface between the C ABI shim (fa_api.cu) and the kernel
// translation units. Host-only declarations; no CUDA types beyond CUtensorMap.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fa {

struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;  // bf16 [BH][N][d], box 64 x 128 x 1, 128B swizzle
  float* lse;                          // fp32 [BH][N]
  unsigned int* status;                // device error word
  int BH, N, d;
  float scale_log2;  // scale * log2(e)
  int causal;
  int head_group;  // heads per CTA scheduling group (set by launch_fwd)
};

struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // bf16 [BH][N][d], box 64 x 128 x 1, 128B swizzle (loads)
  CUtensorMap tm_dq, tm_dk, tm_dv;      // bf16 [BH][N][d], box 64 x 128 x 1, 128B swizzle (stores)
  const void* o;                        // bf16 [BH][N][d]
  const void* dO;                       // bf16 [BH][N][d]
  const float* lse;                     // fp32 [BH][N]
  float* Dsum;                          // fp32 [BH][N], in the caller's workspace
  unsigned int* work;                   // work counters in the caller's workspace ([0] dK/dV, [1] dQ)
  unsigned int* status;
  int BH, N, d;
  float scale, scale_log2;
  int causal;
  int head_group;  // heads per CTA scheduling group (set by launch_bwd)
};

// Heads per CTA scheduling group for a (BH x nblk) grid whose causal CTAs
// cost nblk - blk units of work plus 'overhead' units each (schedule.cu).
int pick_head_group(int BH, int nblk, bool causal, int num_sms, double overhead);

// Each returns cudaSuccess or the launch error.
cudaError_t launch_fwd(const FwdArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_bwd(const BwdArgs& a, int num_sms, cudaStream_t stream);

}  // namespace fa
