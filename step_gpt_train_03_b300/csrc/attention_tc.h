// Causal flash attention for head size 64 on the tcgen05 tensor cores.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>

// 1 when the kernels can run on the current device.
int attention_tc_available();

// out (B,T,C) and lse (B,NH,T) from qkv (B,T,3C); C / NH must be 64, else
// GPT2_EUNSUPPORTED.  `err` (device, nullable) receives the timeout bit.
int attention_tc_forward(cudaStream_t s, __nv_bfloat16* out, float* lse, const __nv_bfloat16* qkv, int B, int T,
                         int C, int NH, unsigned* err);

// dqkv (B,T,3C) [overwritten] from dout (B,T,C), qkv, lse (B,NH,T) and D = rowsum(dout*out)
// (B,NH,T); C / NH must be 64 and T a multiple of 4, else GPT2_EUNSUPPORTED.
int attention_tc_backward(cudaStream_t s, __nv_bfloat16* dqkv, const __nv_bfloat16* dout, const __nv_bfloat16* qkv,
                          const float* lse, const float* D, int B, int T, int C, int NH, unsigned* err);
