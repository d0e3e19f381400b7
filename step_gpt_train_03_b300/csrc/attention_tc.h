// Causal flash attention for head size 64 on the tcgen05 tensor cores.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>

// 1 when the kernels can run on the current device.
int attention_tc_available();

// out (B,T,C) and lse (B,NH,T) from qkv (B,T,3C); C / NH must be 64, else
// GPT2_EUNSUPPORTED.  `err` (device, nullable) receives the timeout bit.
int attention_tc_forward(cudaStream_t s, __nv_bfloat16* out, float* lse, const __nv_bfloat16* qkv, int B, int T,
                         int C, int NH, unsigned* err);

// fp32 scratch elements the backward needs: the row sums D and, for T not a multiple of
// 4, a copy of the LSE, each (B, NH, T rounded up to a multiple of 4).
size_t attention_tc_backward_scratch_floats(int B, int T, int NH);

// dqkv (B,T,3C) [overwritten] from dout (B,T,C), the forward's qkv, out and lse
// (B,NH,T); `scratch` (device, 16-byte aligned, attention_tc_backward_scratch_floats).
// `bias_partial` (device, nullable): receives partial column sums of the stored dqkv,
// row (b * ceil(T/128) + t) * 4 + q of a (B * ceil(T/128) * 4) x 3C fp32 matrix holding
// rows [32q, 32q + 32) of row tile t of batch b; its column sums are the qkv bias
// gradient.  C / NH must be 64, else GPT2_EUNSUPPORTED.
int attention_tc_backward(cudaStream_t s, __nv_bfloat16* dqkv, const __nv_bfloat16* dout, const __nv_bfloat16* qkv,
                          const __nv_bfloat16* out, const float* lse, float* scratch, float* bias_partial, int B,
                          int T, int C, int NH, unsigned* err);

// rows of the bias_partial matrix of attention_tc_backward
static inline int attention_tc_bias_partial_rows(int B, int T) { return B * ((T + 127) / 128) * 4; }
