// bf16 matmuls of the linear layers on the sm_103a tensor cores (tcgen05 + TMEM),
// operands staged by TMA.
//
// ujoy.net llm.c article, section "用C语言实现LLM": the matmul layer's forward and
// backward.  With the weight stored (out, in):
//   forward  y  = x W^T (+ bias, GELU, residual in the epilogue)
//   backward dx = dy W   (GELU backward in the epilogue),  dW += dy^T x
// All three are D[m][n] = sum_k A(m,k) B(n,k) with each operand either K-major
// (row r at ptr + r*ld, k contiguous) or MN-major (k-th row at ptr + k*ld, r
// contiguous); the MMA reads both forms directly (instruction-descriptor major bits),
// so no transposed copies are made.
//
// Kernel: persistent, one CTA per SM, 192 threads.
//   warp 0      TMA producer: 128x64 A tile and BNx64 B tile per stage, 4-stage ring
//   warp 1      TMEM owner and MMA issuer (one thread): 128xBN fp32 accumulator,
//               two accumulators in TMEM so the epilogue of tile i overlaps tile i+1
//   warps 2-5   epilogue: tcgen05.ld 32 rows x 64 columns of the accumulator, fuse
//               bias / GELU / residual / GELU-backward, stage the chunk in a
//               128B-swizzled shared buffer and write it with one TMA store (fp32
//               weight gradients: one TMA reduce-add, so each element is added once);
//               residual and pre-activation inputs arrive by TMA load into the same
//               buffers, one chunk ahead (the next tile's first chunk is requested
//               before its accumulator is ready)
// Every mbarrier wait is bounded: on expiry the kernel raises the timeout bit in the
// library's error word, the other roles see the abort flag and stop, in-flight copies
// and MMAs are waited for (again bounded), TMEM is freed and the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "gemm_simt.cuh"
#include "gemm_tc.h"
#include "runtime.h"
#include "../../include/gpt2.h"

#define TC_BM 128
#define TC_BK 64
#define TC_STAGES 4
#define TC_THREADS 192
#define TC_EPI_PARTIAL 5          // fp32 split-K partial tile into scratch

#include "tc_ptx.cuh"

// ------------------------------------------------------------------ kernel
struct TcEpi {
    void* out;          // bf16 (or fp32 for EPI_ACC_F32 / partial)
    const bf16* bias;   // nullable
    void* aux;          // GELU pre-activation out / residual in / pre-activation in
    long ldo;           // row stride of out and aux (elements)
};

template <int BN>
struct TcSmem {
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;
    static constexpr int B_BYTES = BN * TC_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // two 4 KB staging buffers (32 rows x 128 bytes) per epilogue warp
    static constexpr int STG_OFF = TC_STAGES * STAGE_BYTES;
    static constexpr int STG_BYTES = 4096;
    static constexpr int BAR_OFF = STG_OFF + 4 * 2 * STG_BYTES;
    // full[S], empty[S], acc_full[2], acc_empty[2], done, aux[4 warps][2 buffers];
    // tmem address, abort flag
    static constexpr int TOTAL = BAR_OFF + (2 * TC_STAGES + 13) * 8 + 16 + 1024;
};

// byte offset of 16-byte chunk j of row r in a 128B-swizzled staging buffer
__device__ __forceinline__ int stg_off(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

// D (M x N) over units = m_tiles x n_tiles x splits, n fastest.  Split s of a tile
// covers k-blocks [s*kb_per, min(nkb, (s+1)*kb_per)); partial epilogues write tile
// (s) of the scratch at out + s*M*ldo.
template <int BN, int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmAux, int M, int N,
               int K, int splits, TcEpi ep, unsigned* err) {
    using S = TcSmem<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
    uint64_t* empty = full + TC_STAGES;
    uint64_t* acc_full = empty + TC_STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* done = acc_empty + 2;
    uint64_t* aux_bar = done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux_bar + 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (M + TC_BM - 1) / TC_BM, n_tiles = (N + BN - 1) / BN;
    const int nkb = (K + TC_BK - 1) / TC_BK;
    const int kb_per = (nkb + splits - 1) / splits;
    const int units = m_tiles * n_tiles * splits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < TC_STAGES; i++) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
        for (int i = 0; i < 2; i++) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4); }
        mbar_init(done, 1);
        for (int i = 0; i < 8; i++) mbar_init(&aux_bar[i], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmOut);
        if (EPI == EPI_GELU || EPI == EPI_RESID || EPI == EPI_GELU_BWD) tma_prefetch_desc(&tmAux);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(2 * BN) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const int sp = u % splits, tile = u / splits;
                const int nt = tile % n_tiles, mt = tile / n_tiles;
                const int kb0 = sp * kb_per, kb1 = min(nkb, kb0 + kb_per);
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const int s = it % TC_STAGES;
                    const uint32_t ph = (it / TC_STAGES) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, err)) { ok = false; break; }
                    uint8_t* a = smem + s * S::STAGE_BYTES;
                    uint8_t* b = a + S::A_BYTES;
                    mbar_expect_tx(&full[s], S::STAGE_BYTES);
                    if (!A_MN) {
                        tma_load_2d(a, &tmA, &full[s], kb * TC_BK, mt * TC_BM);
                    } else {
#pragma unroll
                        for (int j = 0; j < TC_BM / 64; j++)
                            tma_load_2d(a + j * 8192, &tmA, &full[s], mt * TC_BM + j * 64, kb * TC_BK);
                    }
                    if (!B_MN) {
                        tma_load_2d(b, &tmB, &full[s], kb * TC_BK, nt * BN);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; j++)
                            tma_load_2d(b + j * 8192, &tmB, &full[s], nt * BN + j * 64, kb * TC_BK);
                    }
                }
            }
            // before leaving, every copy this thread started must have landed
            for (int back = 0; back < TC_STAGES && back < it; back++) {
                const int j = it - 1 - back;
                const long long t0 = clock64();
                while (!mbar_try_wait(&full[j % TC_STAGES], (j / TC_STAGES) & 1))
                    if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16(TC_BM, BN, A_MN, B_MN);
            int it = 0, local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, local++) {
                const int sp = u % splits;
                const int kb0 = sp * kb_per, kb1 = min(nkb, kb0 + kb_per);
                const int acc = local & 1;
                const uint32_t aph = (local >> 1) & 1;
                if (!mbar_wait(&acc_empty[acc], aph ^ 1, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const int s = it % TC_STAGES;
                    const uint32_t ph = (it / TC_STAGES) & 1;
                    if (!mbar_wait(&full[s], ph, abort_flag, err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a = smem_u32(smem + s * S::STAGE_BYTES);
                    const uint32_t b = a + S::A_BYTES;
#pragma unroll
                    for (int k = 0; k < TC_BK / 16; k++) {
                        // K-major: 16 k-elements are 32 bytes inside each 128-byte row;
                        // MN-major: 16 k-rows are two 1024-byte swizzle atoms
                        const uint64_t ad = A_MN ? sdesc(a + k * 2048, 8192, 1024) : sdesc(a + k * 32, 16, 1024);
                        const uint64_t bd = B_MN ? sdesc(b + k * 2048, 8192, 1024) : sdesc(b + k * 32, 16, 1024);
                        tc_mma(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);     // the stage is free once these MMAs have read it
                }
                if (ok) tc_commit(&acc_full[acc]);
            }
            // all MMAs issued by this thread complete before the teardown
            tc_commit(done);
            const long long t0 = clock64();
            while (!mbar_try_wait(done, 0))
                if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
        }
    } else {
        // ---------------------------------------------------------- epilogue warps 2..5
        const int ew = warp - 2;                       // epilogue warp 0..3
        const int lane_grp = warp & 3;                 // TMEM lanes 32*lane_grp .. +31
        uint8_t* stg = smem + S::STG_OFF + ew * 2 * S::STG_BYTES;
        constexpr bool AUX_IN = (EPI == EPI_RESID || EPI == EPI_GELU_BWD);
        constexpr int NCH = BN / 64;                   // 64-column chunks per tile
        uint64_t* auxb = &aux_bar[ew * 2];             // one barrier per staging buffer
        uint32_t aux_ph = 0;                           // bit b: phase of buffer b's barrier
        uint32_t aux_pend = 0;                         // bit b: a load into buffer b not yet waited for
        int nbuf = 0;                                  // staging buffer in use: nbuf & 1
        int local = 0;
        bool alive = true;
        // residual / pre-activation inputs: the load of chunk (unit uu, chunk c) goes to
        // buffer kb once every store still reading a staging buffer has finished
        auto aux_issue = [&](int uu, int c, int kb) {
            if (lane == 0) {
                const int tile = uu / splits;
                const int col = (tile % n_tiles) * BN + c * 64, row0 = (tile / n_tiles) * TC_BM + lane_grp * 32;
                bulk_wait_read<0>();
                aux_pend |= 1u << kb;
                mbar_expect_tx(&auxb[kb], S::STG_BYTES);
                tma_load_2d(stg + kb * S::STG_BYTES, &tmAux, &auxb[kb], col, row0);
            }
        };
        if (AUX_IN && blockIdx.x < units) aux_issue(blockIdx.x, 0, 0);
        for (int u = blockIdx.x; u < units && alive; u += gridDim.x, local++) {
            const int sp = u % splits, tile = u / splits;
            const int nt = tile % n_tiles, mt = tile / n_tiles;
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            // one lane waits; the warp then proceeds converged (tcgen05.ld is warp-wide)
            int okw = 1;
            if (lane == 0) okw = mbar_wait(&acc_full[acc], aph, abort_flag, err) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (!okw) break;
            __syncwarp();
            tc_fence_after();
            const int row0 = mt * TC_BM + lane_grp * 32;   // first of this warp's 32 rows
            const int yout = (EPI == TC_EPI_PARTIAL) ? sp * M + row0 : row0;
#pragma unroll 1
            for (int ci = 0; ci < NCH; ci++) {
                const int c = ci * 64;
                const int col = nt * BN + c;
                if (!AUX_IN && col >= N) break;
                uint32_t r0[32], r1[32];
                const uint32_t ta = tmem_base + ((uint32_t)(lane_grp * 32) << 16) + acc * BN + c;
                tmem_ld32(ta, r0);
                tmem_ld32(ta + 32, r1);
                tmem_ld_wait();
                float v[64];
#pragma unroll
                for (int i = 0; i < 32; i++) { v[i] = __uint_as_float(r0[i]); v[32 + i] = __uint_as_float(r1[i]); }
                if constexpr (EPI == EPI_ACC_F32 || EPI == TC_EPI_PARTIAL) {
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        uint8_t* sb = stg + (nbuf & 1) * S::STG_BYTES;
                        if (lane == 0) bulk_wait_read<1>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 8; j++)
                            *reinterpret_cast<float4*>(sb + stg_off(lane, j)) =
                                make_float4(v[32 * h + 4 * j], v[32 * h + 4 * j + 1], v[32 * h + 4 * j + 2],
                                            v[32 * h + 4 * j + 3]);
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0 && col + 32 * h < N) {
                            if constexpr (EPI == EPI_ACC_F32) tma_reduce_add_2d(&tmOut, sb, col + 32 * h, yout);
                            else tma_store_2d(&tmOut, sb, col + 32 * h, yout);
                            bulk_commit();
                        }
                        nbuf++;
                    }
                } else if constexpr (AUX_IN) {
                    // this chunk's input was loaded into buffer nbuf & 1 ahead of time; start
                    // the next chunk's (or the next tile's first) load into the other buffer
                    const int kb = nbuf & 1;
                    if (ci + 1 < NCH) aux_issue(u, ci + 1, kb ^ 1);
                    else if (u + gridDim.x < units) aux_issue(u + gridDim.x, 0, kb ^ 1);
                    int oka = 1;
                    if (lane == 0) oka = mbar_wait(&auxb[kb], (aux_ph >> kb) & 1, abort_flag, err) ? 1 : 0;
                    oka = __shfl_sync(0xffffffffu, oka, 0);
                    aux_ph ^= 1u << kb;
                    aux_pend &= ~(1u << kb);
                    if (!oka) { alive = false; break; }
                    __syncwarp();
                    uint8_t* sb = stg + kb * S::STG_BYTES;
                    if (ep.bias && EPI == EPI_RESID) {
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            if (col + 8 * q < N) {
                                Vec<bf16> b = load_vec(ep.bias + col + 8 * q);
#pragma unroll
                                for (int e = 0; e < 8; e++) v[8 * q + e] += b.get(e);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        Vec<bf16> a, o;
                        a.v = *reinterpret_cast<const uint4*>(sb + stg_off(lane, j));
#pragma unroll
                        for (int e = 0; e < 8; e++) {
                            if constexpr (EPI == EPI_RESID) o.set(e, v[8 * j + e] + a.get(e));
                            else o.set(e, v[8 * j + e] * gelu_grad_fast(a.get(e)));
                        }
                        *reinterpret_cast<uint4*>(sb + stg_off(lane, j)) = o.v;
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0 && col < N) { tma_store_2d(&tmOut, sb, col, yout); bulk_commit(); }
                    nbuf++;
                } else {
                    if (ep.bias) {
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            if (col + 8 * q < N) {
                                Vec<bf16> b = load_vec(ep.bias + col + 8 * q);
#pragma unroll
                                for (int e = 0; e < 8; e++) v[8 * q + e] += b.get(e);
                            }
                        }
                    }
                    uint8_t* sb = stg + (nbuf & 1) * S::STG_BYTES;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    if constexpr (EPI == EPI_GELU) {
                        // pre-activation out first, then the activation into the other buffer
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            Vec<bf16> o;
#pragma unroll
                            for (int e = 0; e < 8; e++) o.set(e, v[8 * j + e]);
                            *reinterpret_cast<uint4*>(sb + stg_off(lane, j)) = o.v;
#pragma unroll
                            for (int e = 0; e < 8; e++) v[8 * j + e] = gelu_fast(o.get(e));
                        }
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) { tma_store_2d(&tmAux, sb, col, row0); bulk_commit(); }
                        nbuf++;
                        sb = stg + (nbuf & 1) * S::STG_BYTES;
                        if (lane == 0) bulk_wait_read<1>();
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        Vec<bf16> o;
#pragma unroll
                        for (int e = 0; e < 8; e++) o.set(e, v[8 * j + e]);
                        *reinterpret_cast<uint4*>(sb + stg_off(lane, j)) = o.v;
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) { tma_store_2d(&tmOut, sb, col, yout); bulk_commit(); }
                    nbuf++;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
        // every store this warp issued has completed, and no load is still landing in
        // its staging buffers (only possible after an abort), before the CTA retires
        if (lane == 0) {
            bulk_wait<0>();
            for (int kb = 0; kb < 2; kb++) {
                if (!((aux_pend >> kb) & 1)) continue;
                const long long t0 = clock64();
                while (!mbar_try_wait(&auxb[kb], (aux_ph >> kb) & 1))
                    if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
            }
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    __syncwarp();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(2 * BN)
                     : "memory");
}

// out[n][k] += sum_s part[s][n][k], s in order (split-K reduction, deterministic)
__global__ void splitk_reduce_kernel(float* __restrict__ out, const float* __restrict__ part, size_t n4,
                                     int splits) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 acc = reinterpret_cast<float4*>(out)[i];
    for (int s = 0; s < splits; s++) {
        float4 p = reinterpret_cast<const float4*>(part)[(size_t)s * n4 + i];
        acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
    }
    reinterpret_cast<float4*>(out)[i] = acc;
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static int g_num_sms = 0;
static int g_tc_ok = -1;
static std::mutex g_tc_mutex;

int gemm_tc_available() {
    std::lock_guard<std::mutex> lock(g_tc_mutex);
    if (g_tc_ok >= 0) return g_tc_ok;
    g_tc_ok = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return 0;
    if (prop.major != 10) return 0;
    g_num_sms = prop.multiProcessorCount;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return 0;
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    g_tc_ok = 1;
    return 1;
}

// Split-K is only used when a weight gradient has fewer 128x256 tiles than the GPU has
// SMs, with at most 8 splits: its partials never exceed 8 x (SMs x one tile).
#define TC_MAX_SPLITS 8
#define TC_SPLIT_SM_BOUND 160
size_t gemm_tc_scratch_floats(size_t M, size_t N) {
    (void)M;
    (void)N;
    return (size_t)TC_MAX_SPLITS * TC_SPLIT_SM_BOUND * TC_BM * 256;
}

// 2-D tensor map: inner dimension `inner` (contiguous), outer `outer`, row pitch `ld`
// elements of `ebytes` bytes; box {box_inner, box_outer} (box_inner * ebytes = 128);
// 128-byte swizzle; out-of-range reads give zero and out-of-range writes are dropped.
static bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                     uint32_t box_outer, int ebytes = 2) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * ebytes};
    cuuint32_t box[2] = {(cuuint32_t)(128 / ebytes), box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, ebytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

template <int BN, int EPI, bool A_MN, bool B_MN>
static int launch_tc(cudaStream_t s, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                     const CUtensorMap& tx, int M, int N, int K, int splits, const TcEpi& ep, unsigned* err) {
    using SM = TcSmem<BN>;
    static bool attr_set = false;
    auto kern = gemm_tc_kernel<BN, EPI, A_MN, B_MN>;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::TOTAL) != cudaSuccess)
            return GPT2_ECUDA;
        attr_set = true;
    }
    const int units = ((M + TC_BM - 1) / TC_BM) * ((N + BN - 1) / BN) * splits;
    const int grid = units < g_num_sms ? units : g_num_sms;
    kern<<<grid, TC_THREADS, SM::TOTAL, s>>>(ta, tb, to, tx, M, N, K, splits, ep, err);
    rt_note_launches(1);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}

int gemm_tc_forward(cudaStream_t s, bf16* out, const bf16* inp, const bf16* W, const bf16* bias, int M, int N,
                    int K, int epi, bf16* aux, unsigned* err) {
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (N % 8 || K % 8 || M < 1 || !aligned16(out) || !aligned16(inp) || !aligned16(W) ||
        (bias && !aligned16(bias)) || (aux && !aligned16(aux)))
        return GPT2_EUNSUPPORTED;
    CUtensorMap ta, tb, to, tx;
    if (!make_map(&ta, inp, K, M, K, TC_BM) || !make_map(&tb, W, K, N, K, 256) || !make_map(&to, out, N, M, N, 32))
        return GPT2_EUNSUPPORTED;
    if (aux) {
        if (!make_map(&tx, aux, N, M, N, 32)) return GPT2_EUNSUPPORTED;
    } else {
        tx = to;
    }
    TcEpi ep{out, bias, aux, (long)N};
    switch (epi) {
        case EPI_STORE: return launch_tc<256, EPI_STORE, false, false>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        case EPI_GELU: return launch_tc<256, EPI_GELU, false, false>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        case EPI_RESID: return launch_tc<256, EPI_RESID, false, false>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        default: return GPT2_EUNSUPPORTED;
    }
}

int gemm_tc_backward_dx(cudaStream_t s, bf16* dinp, const bf16* dout, const bf16* W, int M, int N, int K, int epi,
                        const bf16* aux, unsigned* err) {
    // dinp (M x K) = dout (M x N) W (N x K): contraction over N; A = dout K-major,
    // B(k_out, n) = W[n][k_out] is MN-major (k_out contiguous)
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (N % 8 || K % 8 || M < 1 || !aligned16(dinp) || !aligned16(dout) || !aligned16(W) ||
        (aux && !aligned16(aux)))
        return GPT2_EUNSUPPORTED;
    CUtensorMap ta, tb, to, tx;
    if (!make_map(&ta, dout, N, M, N, TC_BM) || !make_map(&tb, W, K, N, K, 64) || !make_map(&to, dinp, K, M, K, 32))
        return GPT2_EUNSUPPORTED;
    if (aux) {
        if (!make_map(&tx, aux, K, M, K, 32)) return GPT2_EUNSUPPORTED;
    } else {
        tx = to;
    }
    TcEpi ep{dinp, nullptr, (void*)aux, (long)K};
    if (epi == EPI_GELU_BWD) return launch_tc<256, EPI_GELU_BWD, false, true>(s, ta, tb, to, tx, M, K, N, 1, ep, err);
    if (epi == EPI_STORE) return launch_tc<256, EPI_STORE, false, true>(s, ta, tb, to, tx, M, K, N, 1, ep, err);
    return GPT2_EUNSUPPORTED;
}

static int choose_splits(int tiles, int nkb) {
    // with fewer tiles than SMs, fill the SMs: the split count with the best SM
    // occupancy over whole waves, each split keeping at least 8 k-blocks
    if (tiles >= g_num_sms || g_num_sms > TC_SPLIT_SM_BOUND) return 1;
    int best = 1;
    double best_eff = 0;
    for (int sp = 1; sp <= TC_MAX_SPLITS; sp++) {
        if (sp > 1 && nkb / sp < 8) break;
        const int units = tiles * sp;
        const int waves = (units + g_num_sms - 1) / g_num_sms;
        const double eff = (double)units / (waves * g_num_sms);
        if (eff > best_eff + 1e-9) { best_eff = eff; best = sp; }
    }
    return best;
}

int gemm_tc_backward_dw(cudaStream_t s, float* dW, const bf16* dout, const bf16* inp, int M, int N, int K,
                        float* scratch, size_t scratch_floats, unsigned* err) {
    // dW (N x K) += dout^T (N x M) inp (M x K): contraction over M; A(n, m) = dout[m][n]
    // and B(k, m) = inp[m][k] are both MN-major
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (N % 8 || K % 8 || M < 1 || !aligned16(dW) || !aligned16(dout) || !aligned16(inp))
        return GPT2_EUNSUPPORTED;
    CUtensorMap ta, tb, to;
    if (!make_map(&ta, dout, N, M, N, 64) || !make_map(&tb, inp, K, M, K, 64)) return GPT2_EUNSUPPORTED;
    // 256-wide tiles throughout (measured faster than 128-wide tiles for every weight
    // gradient of the model); split-K fills the GPU when there are fewer tiles than SMs
    const int tiles = ((N + TC_BM - 1) / TC_BM) * ((K + 255) / 256);
    const int nkb = (M + TC_BK - 1) / TC_BK;
    int splits = choose_splits(tiles, nkb);
    // partial tiles of split s are rows [s*N, (s+1)*N) of one map, so a tile must not
    // straddle two splits: N a multiple of the 128-row tile
    if (splits > 1 && (!scratch || (size_t)splits * N * K > scratch_floats || !aligned16(scratch) || N % TC_BM))
        splits = 1;
    if (splits == 1) {
        if (!make_map(&to, dW, K, N, K, 32, 4)) return GPT2_EUNSUPPORTED;
        TcEpi ep{dW, nullptr, nullptr, (long)K};
        return launch_tc<256, EPI_ACC_F32, true, true>(s, ta, tb, to, to, N, K, M, 1, ep, err);
    }
    if (!make_map(&to, scratch, K, (uint64_t)splits * N, K, 32, 4)) return GPT2_EUNSUPPORTED;
    TcEpi ep{scratch, nullptr, nullptr, (long)K};
    int rc = launch_tc<256, TC_EPI_PARTIAL, true, true>(s, ta, tb, to, to, N, K, M, splits, ep, err);
    if (rc != GPT2_OK) return rc;
    const size_t n4 = (size_t)N * K / 4;
    splitk_reduce_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(dW, scratch, n4, splits);
    rt_note_launches(1);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}
