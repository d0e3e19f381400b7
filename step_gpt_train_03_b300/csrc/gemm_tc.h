// bf16 matmuls of the linear layers on the tcgen05 tensor cores (TMA-fed, TMEM
// accumulators).  Each call returns GPT2_EUNSUPPORTED for a shape it does not take (N or
// K not a multiple of 8, an operand not 16-byte aligned, no tcgen05 device); there is no
// other bf16 path.  `err` (device, nullable) is the error word a kernel sets if one of
// its bounded waits runs out.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

// 1 when the tensor-core kernels can run on the current device, else 0.
int gemm_tc_available();

// fp32 scratch elements the dW product may use for split-K partial tiles (M rows of the
// activations, N = its widest output).
size_t gemm_tc_scratch_floats(size_t M, size_t N);

// out (M,N) = inp (M,K) W(N,K)^T + bias, with epilogue epi (EpiKind): aux is the GELU
// pre-activation output (EPI_GELU) or the residual input (EPI_RESID).
// gelu_deriv (EPI_GELU): aux receives gelu'(h) instead of h (for the fused input-gradient
// product of gemm_tc_backward_dx with gelu_deriv).
int gemm_tc_forward(cudaStream_t s, __nv_bfloat16* out, const __nv_bfloat16* inp,
                    const __nv_bfloat16* W, const __nv_bfloat16* bias, int M, int N, int K, int epi,
                    __nv_bfloat16* aux, unsigned* err, bool gelu_deriv = false);

// The same with e4m3 operands (tcgen05 kind::f8f6f4): inp (M,K) and W (N,K) are e4m3 codes,
// row m of inp stands for codes * inp_deq[m] and W for codes * w_deq[0]; the accumulator
// is multiplied by both factors before the epilogue.  K a multiple of 16.
int gemm_tc_forward_fp8(cudaStream_t s, __nv_bfloat16* out, const uint8_t* inp, const float* inp_deq,
                        const uint8_t* W, const float* w_deq, const __nv_bfloat16* bias, int M, int N, int K,
                        int epi, __nv_bfloat16* aux, unsigned* err, bool gelu_deriv = false);

// A plain bf16 product with bf16 output: out (M,N) = sum_k A(m,k) B(n,k), each operand
// K-major (rows of K contiguous) or MN-major (rows of M or N contiguous, K rows); the
// combination (A MN-major, B K-major) is not built.  M, N, K multiples of 8.
// nb such products at once, each operand's nb matrices contiguous (A_l = A + l M K, B_l =
// B + l N K, out_l = out + l M N); for nb > 1, M and N multiples of 256 and K of 64.
int gemm_tc_bf16_batched(cudaStream_t s, __nv_bfloat16* out, const __nv_bfloat16* A, bool a_mn,
                         const __nv_bfloat16* B, bool b_mn, int M, int N, int K, int nb, unsigned* err);
int gemm_tc_bf16(cudaStream_t s, __nv_bfloat16* out, const __nv_bfloat16* A, bool a_mn, const __nv_bfloat16* B,
                 bool b_mn, int M, int N, int K, unsigned* err);

// dinp (M,K) = dout (M,N) W (N,K); epi EPI_STORE or EPI_GELU_BWD (aux = pre-activation).
// csum (nullable, EPI_GELU_BWD only): column sums of the stored dinp over each 32-row
// block, row r of a ceil(M/32) x K fp32 matrix (whose column sums are the bias gradient
// of the layer that produced the pre-activation).  gelu_deriv (EPI_GELU_BWD): aux holds
// gelu'(h) (from gemm_tc_forward with gelu_deriv), dinp = (dout W) * aux.
int gemm_tc_backward_dx(cudaStream_t s, __nv_bfloat16* dinp, const __nv_bfloat16* dout,
                        const __nv_bfloat16* W, int M, int N, int K, int epi, const __nv_bfloat16* aux,
                        float* csum, unsigned* err, bool gelu_deriv = false);

// dW (N,K) fp32 += dout(M,N)^T inp (M,K); with `assign`, dW = the product (the same
// values as adding into zeros).
int gemm_tc_backward_dw(cudaStream_t s, float* dW, const __nv_bfloat16* dout, const __nv_bfloat16* inp,
                        int M, int N, int K, float* scratch, size_t scratch_floats, unsigned* err,
                        bool assign = false);
