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
#include "runtime.h"

#include <algorithm>

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

// Tiles of 128 x 128 outputs, 256 threads with 8 x 8 outputs each (rows ty*4 + i and
// 64 + ty*4 + i, columns likewise, so every shared-memory read is a float4 that the
// warp reads conflict-free), K in steps of SG_BK through two shared-memory buffers:
// the next step's operands are loaded into registers while the current one is
// multiplied.
// When the tiles do not fill the SMs, the contraction is split into S ranges of whole
// K steps: split z writes its fp32 partial tile to scratch and a second kernel adds the
// S partials in order z = 0..S-1 and applies the epilogue (deterministic).  A product
// that neither fills the SMs nor splits (K too short, no scratch) runs on 64 x 64 tiles.
#define SG_BM 128
#define SG_BN 128
#ifndef SG_BK
#define SG_BK 16                  // 124M fp32 B4 T64 step: 8.75 ms; 9.40 at 8, 8.97 at 32
#endif
#define SG_NL (SG_BK / 8)         // 16-byte packets per thread per operand and K step
#define SG_PAD 4                  // row padding: conflict-free transposed stores
#define SG_THREADS 256
#define SG_MAX_SPLITS 32
#ifndef SG_SPLIT_BLOCKS
#define SG_SPLIT_BLOCKS 4         // blocks per SM that the splits aim for
#endif

// One K step of a 128-row operand tile: SG_NL packets of 4 elements per thread, packet
// e = t + 256 l.  K-contiguous source (X[r * ld + k]): row e / (SG_BK / 4), k =
// 4 (e % (SG_BK / 4)) .. +3; R-contiguous source (X[k * ld + r]): k = e / 32, rows
// 4 (e % 32) .. +3.  VEC: 16-byte loads (the caller checked alignment, ld % 4 and the
// contiguous extent % 4); elements past R or K are 0.
template <typename T, bool KC, bool VEC>
__device__ __forceinline__ void sg_load(const T* __restrict__ X, long ld, int r0, int R, int k0, int K, int t,
                                        float (&v)[SG_NL][4]) {
#pragma unroll
    for (int l = 0; l < SG_NL; l++) {
        const int e = t + SG_THREADS * l;
        const int r = r0 + (KC ? e / (SG_BK / 4) : 4 * (e % 32));
        const int k = k0 + (KC ? 4 * (e % (SG_BK / 4)) : e / 32);
        if constexpr (VEC) {
            float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < R && k < K)
                q = *reinterpret_cast<const float4*>(X + (KC ? (size_t)r * ld + k : (size_t)k * ld + r));
            v[l][0] = q.x; v[l][1] = q.y; v[l][2] = q.z; v[l][3] = q.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int ri = KC ? r : r + i, ki = KC ? k + i : k;
                v[l][i] = (ri < R && ki < K) ? to_f32(X[KC ? (size_t)ri * ld + ki : (size_t)ki * ld + ri]) : 0.f;
            }
        }
    }
}
template <bool KC>
__device__ __forceinline__ void sg_store(float (*S)[SG_BM + SG_PAD], int t, const float (&v)[SG_NL][4]) {
#pragma unroll
    for (int l = 0; l < SG_NL; l++) {
        const int e = t + SG_THREADS * l;
        if constexpr (KC) {
            const int r = e / (SG_BK / 4), k = 4 * (e % (SG_BK / 4));
#pragma unroll
            for (int i = 0; i < 4; i++) S[k + i][r] = v[l][i];
        } else {
            *reinterpret_cast<float4*>(&S[e / 32][4 * (e % 32)]) = make_float4(v[l][0], v[l][1], v[l][2], v[l][3]);
        }
    }
}

// part (nullable): split z of gridDim.z writes its partial tile to part + z*M*N
// (row pitch N) instead of applying the epilogue
template <typename T, bool A_KC, bool B_KC, bool VEC, int EPI>
__global__ void __launch_bounds__(SG_THREADS, 2)
gemm_simt_kernel(const T* __restrict__ A, const T* __restrict__ B, int M, int N, int K,
                 long lda, long ldb, EpiArgs ep, float* __restrict__ part) {
    pdl_wait();
    __shared__ __align__(16) float As[2][SG_BK][SG_BM + SG_PAD];
    __shared__ __align__(16) float Bs[2][SG_BK][SG_BN + SG_PAD];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
    const int nk = (K + SG_BK - 1) / SG_BK;
    const int kt0 = (int)((long)nk * blockIdx.z / gridDim.z), kt1 = (int)((long)nk * (blockIdx.z + 1) / gridDim.z);
    float acc[8][8] = {};
    float ra[SG_NL][4], rb[SG_NL][4];
    if (kt0 < kt1) {
        sg_load<T, A_KC, VEC>(A, lda, m0, M, kt0 * SG_BK, K, tid, ra);
        sg_load<T, B_KC, VEC>(B, ldb, n0, N, kt0 * SG_BK, K, tid, rb);
        sg_store<A_KC>(As[0], tid, ra);
        sg_store<B_KC>(Bs[0], tid, rb);
    }
    __syncthreads();
    for (int kt = kt0; kt < kt1; kt++) {
        const int cur = (kt - kt0) & 1;
        const bool more = kt + 1 < kt1;
        if (more) {                                   // next step's operands, in flight during the FMAs
            sg_load<T, A_KC, VEC>(A, lda, m0, M, (kt + 1) * SG_BK, K, tid, ra);
            sg_load<T, B_KC, VEC>(B, ldb, n0, N, (kt + 1) * SG_BK, K, tid, rb);
        }
#pragma unroll
        for (int kk = 0; kk < SG_BK; kk++) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][kk][64 + tx * 4]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 8; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        if (more) {
            sg_store<A_KC>(As[cur ^ 1], tid, ra);
            sg_store<B_KC>(Bs[cur ^ 1], tid, rb);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (m >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int nb = n0 + h * 64 + tx * 4;
            if (part) {
                float* pr = part + ((size_t)blockIdx.z * M + m) * N;
                if (VEC && nb + 3 < N && (N & 3) == 0) {
                    *reinterpret_cast<float4*>(pr + nb) =
                        make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        if (nb + j < N) pr[nb + j] = acc[i][4 * h + j];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; j++)
                    if (nb + j < N) epi_apply<T, EPI>(ep, m, nb + j, acc[i][4 * h + j]);
            }
        }
    }
}

// Products too small to fill the SMs and too short to split: 64 x 64 tiles, 4 x 4
// outputs per thread, K in steps of 16 (more blocks, shorter chains per thread).
#define SGS_BM 64
#define SGS_BN 64
#define SGS_BK 16
template <typename T, bool A_KC, bool B_KC, int EPI>
__global__ void __launch_bounds__(SG_THREADS)
gemm_simt_small_kernel(const T* __restrict__ A, const T* __restrict__ B, int M, int N, int K,
                 long lda, long ldb, EpiArgs ep) {
    pdl_wait();
    __shared__ float As[SGS_BK][SGS_BM + 4];
    __shared__ float Bs[SGS_BK][SGS_BN + 4];
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * SGS_BM, n0 = blockIdx.x * SGS_BN;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += SGS_BK) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            int e = tid + SG_THREADS * i;
            int mm, kk;
            if (A_KC) { mm = e / SGS_BK; kk = e % SGS_BK; } else { kk = e / SGS_BM; mm = e % SGS_BM; }
            int gm = m0 + mm, gk = k0 + kk;
            float a = 0.f;
            if (gm < M && gk < K) a = to_f32(A_KC ? A[(size_t)gm * lda + gk] : A[(size_t)gk * lda + gm]);
            As[kk][mm] = a;
            int nn;
            if (B_KC) { nn = e / SGS_BK; kk = e % SGS_BK; } else { kk = e / SGS_BN; nn = e % SGS_BN; }
            int gn = n0 + nn;
            gk = k0 + kk;
            float b = 0.f;
            if (gn < N && gk < K) b = to_f32(B_KC ? B[(size_t)gn * ldb + gk] : B[(size_t)gk * ldb + gn]);
            Bs[kk][nn] = b;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SGS_BK; kk++) {
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


// The S partial tiles added in order, then the epilogue (one thread per output)
template <typename T, int EPI>
__global__ void __launch_bounds__(256) gemm_simt_splitk_reduce(const float* __restrict__ part, int S, int M, int N,
                                                               EpiArgs ep) {
    pdl_wait();
    const size_t MN = (size_t)M * N;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= MN) return;
    float acc = part[idx];
    for (int z = 1; z < S; z++) acc += part[z * MN + idx];
    epi_apply<T, EPI>(ep, (int)(idx / N), (int)(idx % N), acc);
}

// SM count of the device current at the first call: it only steers the split choice
static int sg_num_sms() {
    static const int n = [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            return 148;
        return v;
    }();
    return n;
}

// Contraction splits: about SG_SPLIT_BLOCKS blocks per SM when the tiles alone give
// fewer, each split at least 128 of K, bounded by the scratch (S partial M x N tiles)
static int sg_splits(int M, int N, int K, size_t scratch_floats) {
    const long tiles = (long)((M + SG_BM - 1) / SG_BM) * ((N + SG_BN - 1) / SG_BN);
    const long want = (long)SG_SPLIT_BLOCKS * sg_num_sms();
    if (tiles >= want || scratch_floats == 0) return 1;
    long S = (want + tiles - 1) / tiles;
    S = std::min<long>(S, K / 128);
    S = std::min<long>(S, SG_MAX_SPLITS);
    S = std::min<long>(S, (long)(scratch_floats / ((size_t)M * N)));
    return S > 1 ? (int)S : 1;
}

// scratch (device fp32, nullable): room for split partial tiles
template <typename T, bool A_KC, bool B_KC, int EPI>
static cudaError_t launch_gemm_simt(cudaStream_t s, const T* A, long lda, const T* B, long ldb,
                                    int M, int N, int K, const EpiArgs& ep, float* scratch = nullptr,
                                    size_t scratch_floats = 0) {
    // 16-byte loads when every row start is 16-byte aligned and the contiguous extents
    // are whole float4s (fp32 only)
    const bool vec = sizeof(T) == 4 && ((uintptr_t)A & 15) == 0 && ((uintptr_t)B & 15) == 0 && lda % 4 == 0 &&
                     ldb % 4 == 0 && (A_KC ? K : M) % 4 == 0 && (B_KC ? K : N) % 4 == 0 &&
                     ((uintptr_t)scratch & 15) == 0;
    const int S = sg_splits(M, N, K, scratch ? scratch_floats : 0);
    const long tiles = (long)ceil_div(M, SG_BM) * ceil_div(N, SG_BN);
    if (S == 1 && tiles < sg_num_sms()) {
        dim3 grid(ceil_div(N, SGS_BN), ceil_div(M, SGS_BM));
        launch_pdl(gemm_simt_small_kernel<T, A_KC, B_KC, EPI>, grid, SG_THREADS, 0, s, A, B, M, N, K, lda, ldb, ep);
        return cudaGetLastError();
    }
    float* part = S > 1 ? scratch : nullptr;
    dim3 grid(ceil_div(N, SG_BN), ceil_div(M, SG_BM), S);
    if (vec) launch_pdl(gemm_simt_kernel<T, A_KC, B_KC, true, EPI>, grid, SG_THREADS, 0, s, A, B, M, N, K, lda, ldb, ep, part);
    else launch_pdl(gemm_simt_kernel<T, A_KC, B_KC, false, EPI>, grid, SG_THREADS, 0, s, A, B, M, N, K, lda, ldb, ep, part);
    if (S > 1) {
        const size_t MN = (size_t)M * N;
        launch_pdl(gemm_simt_splitk_reduce<T, EPI>, dim3((unsigned)((MN + 255) / 256)), 256, 0, s, (const float*)part, S, M,
                   N, ep);
        rt_note_launches(1);
    }
    return cudaGetLastError();
}
