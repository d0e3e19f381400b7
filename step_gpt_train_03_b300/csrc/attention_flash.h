// bf16 causal attention that keeps only the log-sum-exp of each score row (no T x T
// matrix in memory); the backward recomputes the probabilities from q, k and the LSE.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>

// out (B,T,C) = causal softmax(q k^T / sqrt(hs)) v per head; lse (B,NH,T) fp32.
// `err` (device, nullable) receives the timeout bit of the tensor-core kernel.
int attention_flash_forward(cudaStream_t s, __nv_bfloat16* out, float* lse, const __nv_bfloat16* qkv,
                            int B, int T, int C, int NH, unsigned* err);

// dqkv (B,T,3C) from dout (B,T,C), qkv, out and lse.  scratch holds (B,NH,T) fp32
// row sums D = rowsum(dout * out).
int attention_flash_backward(cudaStream_t s, __nv_bfloat16* dqkv, const __nv_bfloat16* dout,
                             const __nv_bfloat16* qkv, const __nv_bfloat16* out, const float* lse,
                             float* scratch, int B, int T, int C, int NH, unsigned* err);
