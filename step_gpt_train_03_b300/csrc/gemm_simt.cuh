// FMA (SIMT) matmul with fused epilogues: the fp32 path's contraction, where every
// product and sum stays in fp32 so the step matches an fp32 CPU program to rounding.
//
// C(m,n) = sum_k A(m,k) B(n,k), fp32 accumulation.  A is K-contiguous (A[m*lda + k]) or
// M-contiguous (A[k*lda + m]); B likewise.  The three products of a linear layer
// (ujoy.net llm.c article, section "用C语言实现LLM": matmul forward and backward) map to
//   forward  y  = x W^T   : A = x (K-contig), B = W (K-contig)
//   backward dx = dy W    : A = dy (K-contig), B(n,k) = W[k][n] (N-contig)
//   backward dW += dy^T x : A(m,k) = dy[k][m], B(n,k) = x[k][n] (both M/N-contig)
#pragma once
#include "common.cuh"

enum EpiKind {
    EPI_STORE = 0,     // out = acc (+ bias)
    EPI_GELU = 1,      // aux = acc + bias (pre-activation); out = gelu(aux)
    EPI_RESID = 2,     // out = resid + acc + bias          (resid read from aux)
    EPI_GELU_BWD = 3,  // out = acc * gelu'(aux)            (aux = pre-activation)
    EPI_ACC_F32 = 4    // outf[m][n] += acc                 (fp32 parameter grads)
};

struct EpiArgs {
    void* out;          // T* (float* for EPI_ACC_F32)
    const void* bias;   // T*, nullable
    void* aux;          // see EpiKind
    long ldo;           // row stride of out and aux, elements
};

template <typename T, int EPI>
__device__ __forceinline__ void epi_apply(const EpiArgs& ep, int m, int n, float acc) {
    size_t o = (size_t)m * ep.ldo + n;
    if constexpr (EPI == EPI_ACC_F32) {
        float* out = reinterpret_cast<float*>(ep.out);
        out[o] += acc;
    } else {
        T* out = reinterpret_cast<T*>(ep.out);
        float bias = ep.bias ? to_f32(reinterpret_cast<const T*>(ep.bias)[n]) : 0.f;
        if constexpr (EPI == EPI_STORE) {
            out[o] = from_f32<T>(acc + bias);
        } else if constexpr (EPI == EPI_GELU) {
            T pre = from_f32<T>(acc + bias);
            reinterpret_cast<T*>(ep.aux)[o] = pre;
            out[o] = from_f32<T>(gelu_f(to_f32(pre)));
        } else if constexpr (EPI == EPI_RESID) {
            float r = to_f32(reinterpret_cast<const T*>(ep.aux)[o]);
            out[o] = from_f32<T>(r + (acc + bias));
        } else if constexpr (EPI == EPI_GELU_BWD) {
            float pre = to_f32(reinterpret_cast<const T*>(ep.aux)[o]);
            out[o] = from_f32<T>(acc * gelu_grad_f(pre));
        }
    }
}

#define SG_BM 64
#define SG_BN 64
#define SG_BK 16
#define SG_THREADS 256
template <typename T, bool A_KC, bool B_KC, int EPI>
__global__ void __launch_bounds__(SG_THREADS)
gemm_simt_kernel(const T* __restrict__ A, const T* __restrict__ B, int M, int N, int K,
                 long lda, long ldb, EpiArgs ep) {
    pdl_wait();
    __shared__ float As[SG_BK][SG_BM + 4];
    __shared__ float Bs[SG_BK][SG_BN + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += SG_BK) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int e = tid + SG_THREADS * i;
            int mm, kk;
            if (A_KC) { mm = e / SG_BK; kk = e % SG_BK; } else { kk = e / SG_BM; mm = e % SG_BM; }
            int gm = m0 + mm, gk = k0 + kk;
            float a = 0.f;
            if (gm < M && gk < K) a = to_f32(A_KC ? A[(size_t)gm * lda + gk] : A[(size_t)gk * lda + gm]);
            As[kk][mm] = a;
            int nn;
            if (B_KC) { nn = e / SG_BK; kk = e % SG_BK; } else { kk = e / SG_BN; nn = e % SG_BN; }
            int gn = n0 + nn;
            gk = k0 + kk;
            float b = 0.f;
            if (gn < N && gk < K) b = to_f32(B_KC ? B[(size_t)gn * ldb + gk] : B[(size_t)gk * ldb + gn]);
            Bs[kk][nn] = b;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SG_BK; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) { a[i] = As[kk][ty + 16 * i]; b[i] = Bs[kk][tx + 16 * i]; }
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int m = m0 + ty + 16 * i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int n = n0 + tx + 16 * j;
            if (n < N) epi_apply<T, EPI>(ep, m, n, acc[i][j]);
        }
    }
}

template <typename T, bool A_KC, bool B_KC, int EPI>
static cudaError_t launch_gemm_simt(cudaStream_t s, const T* A, long lda, const T* B, long ldb,
                                    int M, int N, int K, const EpiArgs& ep) {
    dim3 grid(ceil_div(N, SG_BN), ceil_div(M, SG_BM));
    launch_pdl(gemm_simt_kernel<T, A_KC, B_KC, EPI>, grid, SG_THREADS, 0, s, A, B, M, N, K, lda, ldb, ep);
    return cudaGetLastError();
}
