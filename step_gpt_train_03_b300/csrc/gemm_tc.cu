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
// Kernel: persistent, one CTA per SM, 320 threads; large products run on CTA pairs
// (2-CTA clusters, 256 x 256 tiles, tcgen05 cta_group::2: each CTA stages half of B and
// reads half the operand bytes per MMA).
//   warp 0      TMA producer: 128x64 A tile and BNx64 B tile per stage, 4-stage ring
//   warp 1      TMEM owner and MMA issuer (one thread): 128xBN fp32 accumulator,
//               two accumulators in TMEM so the epilogue of tile i overlaps tile i+1
//   warps 2-9   epilogue, two warps per TMEM lane quadrant (warp w reads lanes
//               32*(w%4)..+31), each taking half of the tile's columns: tcgen05.ld
//               32 rows x 64 columns of the accumulator, fuse bias / GELU / residual /
//               GELU-backward, stage 32-column pieces in 64B-swizzled 2 KB shared
//               buffers and write each with one TMA store (fp32 weight gradients: one
//               TMA reduce-add, so each element is added once); residual and
//               pre-activation inputs arrive by TMA load into the same buffers, one
//               piece ahead (the next tile's first piece is requested before its
//               accumulator is ready)
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
#define TC_EPI_WARPS 8
#define TC_THREADS (64 + 32 * TC_EPI_WARPS)
#define TC_EPI_PARTIAL 5          // fp32 split-K partial tile into scratch
#ifndef TC_PAIR_NACC
#define TC_PAIR_NACC 2            // TMEM accumulators of a CTA pair
#endif

#include "tc_ptx.cuh"

// ------------------------------------------------------------------ kernel
struct TcEpi {
    void* out;          // bf16 (or fp32 for EPI_ACC_F32 / partial)
    const bf16* bias;   // nullable
    void* aux;          // GELU pre-activation out / residual in / pre-activation in
    long ldo;           // row stride of out and aux (elements)
    const float* a_deq; // e4m3 products: per-row unscaling factor of A (M floats)
    const float* b_deq; // e4m3 products: unscaling factor of B (one float)
    float* csum;        // GELU backward (nullable): column sums of the stored output over
                        // each 32-row block, row r of a ceil(M/32) x N fp32 matrix
    // batched products (nb > 1): nb independent products whose operands and outputs are
    // stacked along the rows of their tensor maps, batch element l's rows starting at
    // l * a_rows (A), l * b_rows (B), l * o_rows (out)
    int nb, a_rows, b_rows, o_rows;
    // GELU epilogues: with gelu_deriv the forward keeps gelu'(h) instead of h in aux, and
    // the input-gradient product multiplies by aux as it is (already the derivative)
    int gelu_deriv;
};

// Staging buffers per epilogue warp: four for the GELU epilogues of a CTA pair (two
// stores per piece forward, a load ahead of each store backward, so two buffers leave
// the warp waiting on its own stores), else two.
template <int EPI, int CL>
struct TcBufs {
    static constexpr int value = (CL == 2 && (EPI == EPI_GELU || EPI == EPI_GELU_BWD)) ? 4 : 2;
};

// CL = 1: one CTA holds a 128 x 64 A and a BN x 64 B block per stage, 4 stages.
// CL = 2 (CTA pair): each CTA holds its 128 x 64 A block and half of the B block, so a
// stage is 2/3 the size and 6 stages fit (5 with four staging buffers per warp).
template <int BN, int CL = 1, int NB = 2>
struct TcSmem {
    static constexpr int STAGES = CL == 2 ? (NB > 2 ? 5 : 6) : TC_STAGES;
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;
    static constexpr int B_BYTES = BN / CL * TC_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // NB 2 KB staging buffers (32 rows x 64 bytes) per epilogue warp
    static constexpr int STG_OFF = STAGES * STAGE_BYTES;
    static constexpr int STG_BYTES = 2048;
    static constexpr int BAR_OFF = STG_OFF + TC_EPI_WARPS * NB * STG_BYTES;
    // full[S], empty[S], acc_full[2], acc_empty[2], done, aux[epilogue warps][NB buffers];
    // tmem address, abort flag
    static constexpr int NBAR = 2 * STAGES + 5 + NB * TC_EPI_WARPS;
    static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16 + 1024;
    static_assert(TOTAL <= 232448, "shared memory of one CTA");
    static_assert(NB == 2 || NB == 4, "staging ring");
};

// byte offset of 16-byte unit j (0..3) of row r in a 64B-swizzled staging buffer of
// 64-byte rows: the unit index is XORed with bits 1-2 of the row, so the 32 rows of a
// warp's 16-byte store fall on distinct bank groups in each quarter-warp phase
__device__ __forceinline__ int stg_off(int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) << 4); }

// D (M x N) over units = m_groups x n_tiles x splits, where a group is CL consecutive
// 128-row tiles; units run n fastest, or m fastest when B is the larger operand (each B
// tile is then read once while all of A stays in L2).  Split s of a tile covers k-blocks [s*kb_per, min(nkb,
// (s+1)*kb_per)); partial epilogues write tile (s) of the scratch at out + s*M*ldo.
// CL = 2: the two CTAs of a cluster are a CTA pair computing one 256 x BN tile with
// 256-row MMAs issued by the leader (rank 0) on both CTAs' tensor cores.  Each CTA
// loads its own 128 A rows and its half of the B columns; all loads count on the
// leader's full barrier; the leader's commits release the stage and announce the
// accumulator in both CTAs; each CTA's epilogue drains its own 128 rows of TMEM and
// frees the accumulator on the leader's barrier.  Per CTA this halves the B operand
// reads and shared-memory traffic of each MMA.  NACC accumulators of BN columns.
// F8: e4m3 operands (kind::f8f6f4, K-major A and B only): a k-block is 128 elements, so
// every byte offset, box and descriptor is that of the bf16 kernel; the epilogue
// multiplies the accumulator by the row's A factor times the B factor.
template <int BN, int EPI, bool A_MN, bool B_MN, int CL = 1, bool F8 = false>
__global__ void __launch_bounds__(TC_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmAux, int M, int N,
               int K, int splits, int m_fast, TcEpi ep, unsigned* err) {
    constexpr int NB = TcBufs<EPI, CL>::value;
    using S = TcSmem<BN, CL, NB>;
    constexpr int STAGES = S::STAGES;
    constexpr int NACC = CL == 2 ? TC_PAIR_NACC : 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* done = acc_empty + 2;
    uint64_t* aux_bar = done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux_bar + NB * TC_EPI_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (M + TC_BM - 1) / TC_BM, n_tiles = (N + BN - 1) / BN;
    constexpr int BKE = F8 ? 2 * TC_BK : TC_BK;        // elements per k-block (128 bytes)
    static_assert(!F8 || (!A_MN && !B_MN), "e4m3 operands are K-major");
    const int nkb = (K + BKE - 1) / BKE;
    const int kb_per = (nkb + splits - 1) / splits;
    const int m_groups = (m_tiles + CL - 1) / CL;
    const int nbat = ep.nb > 1 ? ep.nb : 1;
    const int upb = m_groups * n_tiles * splits;        // units per batch element
    const int units = upb * nbat;
    const int crank = CL > 1 ? (int)cluster_rank() : 0;
    const bool leader = crank == 0;
    const int ustart = blockIdx.x / CL, ustep = gridDim.x / CL;    // this cluster's units
    constexpr uint16_t CMASK = (1u << CL) - 1;
    // unit -> (split, m tile, n tile) of batch element u / upb (upb is a multiple of
    // splits, so u % splits is the split in every role)
    auto decode = [&](int u, int& sp, int& mt, int& nt, int& lb) {
        lb = u / upb;
        u -= lb * upb;
        sp = u % splits;
        const int tile = u / splits;
        const int mg = m_fast ? tile % m_groups : tile / n_tiles;
        nt = m_fast ? tile / m_groups : tile % n_tiles;
        mt = mg * CL + crank;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; i++) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
        for (int i = 0; i < 2; i++) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], CL * TC_EPI_WARPS); }
        mbar_init(done, 1);
        for (int i = 0; i < NB * TC_EPI_WARPS; i++) mbar_init(&aux_bar[i], 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmOut);
        if (EPI == EPI_GELU || EPI == EPI_RESID || EPI == EPI_GELU_BWD) tma_prefetch_desc(&tmAux);
    }
    if (warp == 1) {
        if constexpr (CL == 1) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(smem_u32(tmem_slot)), "r"(NACC * BN) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        } else {
            // one warp of each CTA of the pair: the same columns in both CTAs' TMEM
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                         ::"r"(smem_u32(tmem_slot)), "r"(NACC * BN) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if (CL > 1) cluster_sync();        // the peer's barriers and TMEM address exist from here on
    tc_fence_after();
    // set-up done (barriers, TMEM, descriptor prefetch): wait for the predecessor's
    // results, and let the next kernel's CTAs launch onto SMs as ours retire
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem_base = *tmem_slot;
    // the pair's MMAs write one TMEM address in both CTAs: if the two allocations
    // differ, no work is done (both CTAs see the same two values and agree)
    bool pair_ok = true;
    if (CL > 1) {
        pair_ok = ld_shared_cluster_u32(mapa_shared(tmem_slot, (uint32_t)(crank ^ 1))) == tmem_base;
        if (!pair_ok && threadIdx.x == 0) raise_error(err, ERRBIT_TIMEOUT);
    }
    const int ufirst = pair_ok ? ustart : units;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            const uint32_t full_lead = CL > 1 ? mapa_shared(full, 0) : 0;   // the leader's full[0]
            constexpr int BH = BN / CL;                                      // B rows (or columns) per CTA
            for (int u = ufirst; u < units && ok; u += ustep) {
                int sp, mt, nt, lb;
                decode(u, sp, mt, nt, lb);
                const int kb0 = sp * kb_per, kb1 = min(nkb, kb0 + kb_per);
                const int nb0 = nt * BN + crank * BH;                        // first B row of this CTA's share
                const int ay = lb * ep.a_rows, by = lb * ep.b_rows;          // batch element's first rows
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, err)) { ok = false; break; }
                    uint8_t* a = smem + s * S::STAGE_BYTES;
                    uint8_t* b = a + S::A_BYTES;
                    if constexpr (CL == 1) {
                        mbar_expect_tx(&full[s], S::STAGE_BYTES);
                        if (!A_MN) {
                            tma_load_2d(a, &tmA, &full[s], kb * BKE, ay + mt * TC_BM);
                        } else {
#pragma unroll
                            for (int j = 0; j < TC_BM / 64; j++)
                                tma_load_2d(a + j * 8192, &tmA, &full[s], mt * TC_BM + j * 64, ay + kb * BKE);
                        }
                        if (!B_MN) {
                            tma_load_2d(b, &tmB, &full[s], kb * BKE, by + nb0);
                        } else {
#pragma unroll
                            for (int j = 0; j < BN / 64; j++)
                                tma_load_2d(b + j * 8192, &tmB, &full[s], nb0 + j * 64, by + kb * BKE);
                        }
                    } else {
                        // both CTAs' bytes are counted on the leader's barrier
                        const uint32_t fb = full_lead + s * 8;
                        if (leader) mbar_expect_tx(&full[s], CL * S::STAGE_BYTES);
                        if (!A_MN) {
                            tma_load_2d_pair(a, &tmA, fb, kb * BKE, ay + mt * TC_BM);
                        } else {
#pragma unroll
                            for (int j = 0; j < TC_BM / 64; j++)
                                tma_load_2d_pair(a + j * 8192, &tmA, fb, mt * TC_BM + j * 64, ay + kb * BKE);
                        }
                        if (!B_MN) {
                            tma_load_2d_pair(b, &tmB, fb, kb * BKE, by + nb0);
                        } else {
#pragma unroll
                            for (int j = 0; j < BH / 64; j++)
                                tma_load_2d_pair(b + j * 8192, &tmB, fb, nb0 + j * 64, by + kb * BKE);
                        }
                    }
                }
            }
            // before leaving, every copy this CTA's barriers count must have landed (in a
            // pair the leader's barriers count both CTAs' copies)
            if (CL == 1 || leader) {
                for (int back = 0; back < STAGES && back < it; back++) {
                    const int j = it - 1 - back;
                    const long long t0 = clock64();
                    while (!mbar_try_wait(&full[j % STAGES], (j / STAGES) & 1))
                        if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
                }
            }
            // and, in a pair, every release of the last stages (the leader's commits) must
            // have arrived on this CTA's barriers
            if (CL > 1) {
                for (int back = 0; back < STAGES && back < it; back++) {
                    const int j = it - 1 - back;
                    const long long t0 = clock64();
                    while (!mbar_try_wait(&empty[j % STAGES], (j / STAGES) & 1))
                        if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // (in a pair only the leader's thread issues; its MMAs drive both tensor cores)
        if (lane == 0 && (CL == 1 || leader)) {
            constexpr uint32_t IDESC = F8 ? idesc_e4m3(TC_BM * CL, BN, A_MN, B_MN) : idesc_bf16(TC_BM * CL, BN, A_MN, B_MN);
            int it = 0, local = 0;
            bool ok = true;
            for (int u = ufirst; u < units && ok; u += ustep, local++) {
                const int sp = u % splits;
                const int kb0 = sp * kb_per, kb1 = min(nkb, kb0 + kb_per);
                const int acc = local % NACC;
                const uint32_t aph = (local / NACC) & 1;
                if (!mbar_wait(&acc_empty[acc], aph ^ 1, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
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
                        const uint32_t accf = (kb > kb0 || k > 0) ? 1u : 0u;
                        if constexpr (F8) {
                            if constexpr (CL == 1) tc_mma_f8(d_tmem, ad, bd, IDESC, accf);
                            else tc_mma_pair_f8(d_tmem, ad, bd, IDESC, accf);
                        } else {
                            if constexpr (CL == 1) tc_mma(d_tmem, ad, bd, IDESC, accf);
                            else tc_mma_pair(d_tmem, ad, bd, IDESC, accf);
                        }
                    }
                    // the stage is free (in both CTAs of a pair) once these MMAs have read it
                    if constexpr (CL == 1) tc_commit(&empty[s]);
                    else tc_commit_pair_mc(&empty[s], CMASK);
                }
                if (ok) {
                    if constexpr (CL == 1) tc_commit(&acc_full[acc]);
                    else tc_commit_pair_mc(&acc_full[acc], CMASK);
                }
            }
            // all MMAs issued by this thread complete before the teardown
            if constexpr (CL == 1) tc_commit(done);
            else tc_commit_pair(done);
            const long long t0 = clock64();
            while (!mbar_try_wait(done, 0))
                if (clock64() - t0 > TC_WAIT_LIMIT) { raise_error(err, ERRBIT_TIMEOUT); break; }
        }
    } else {
        // ---------------------------------------------------------- epilogue warps 2..9
        const int ew = warp - 2;                       // epilogue warp 0..7
        const int lane_grp = warp & 3;                 // TMEM lanes 32*lane_grp .. +31
        const int cbase = (ew >> 2) * (BN / 2);        // this warp's half of the tile's columns
        uint8_t* stg = smem + S::STG_OFF + ew * NB * S::STG_BYTES;
        constexpr bool AUX_IN = (EPI == EPI_RESID || EPI == EPI_GELU_BWD);
        constexpr int NPAIR = BN / 128;                // 64-column accumulator loads per warp per tile
        constexpr int NPC = 2 * NPAIR;                 // 32-column pieces per warp per tile
        constexpr int AHEAD = NB / 2;                  // input pieces loaded ahead of the one in use
        uint64_t* auxb = &aux_bar[ew * NB];            // one barrier per staging buffer
        uint32_t aux_ph = 0;                           // bit b: phase of buffer b's barrier
        uint32_t aux_pend = 0;                         // bit b: a load into buffer b not yet waited for
        int nbuf = 0;                                  // staging buffer in use: nbuf % NB
        int local = 0;
        bool alive = true;
        // residual / pre-activation inputs: with inputs, every tile of this warp is NPC
        // pieces and piece g uses buffer g % NB.  The load of piece g goes out once the
        // store of piece g - NB (the buffer's last user) has read it; the stores of the
        // pieces after that one may still be in flight.
        auto aux_issue = [&](int g) {
            const int uu = ufirst + (g / NPC) * ustep, pc = g % NPC, kb = g % NB;
            if (lane == 0 && uu < units) {
                int usp, umt, unt, ulb;
                decode(uu, usp, umt, unt, ulb);
                const int col = unt * BN + cbase + pc * 32;
                const int row0 = ulb * ep.o_rows + umt * TC_BM + lane_grp * 32;
                bulk_wait_read<NB - AHEAD - 1>();
                aux_pend |= 1u << kb;
                mbar_expect_tx(&auxb[kb], S::STG_BYTES);
                tma_load_2d(stg + kb * S::STG_BYTES, &tmAux, &auxb[kb], col, row0);
            }
        };
        // bias (nullable) added to 32 columns starting at global column col
        auto add_bias = [&](float* v, int col) {
            if (ep.bias) {
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    if (col + 8 * q < N) {
                        Vec<bf16> b = load_vec(ep.bias + col + 8 * q);
#pragma unroll
                        for (int e = 0; e < 8; e++) v[8 * q + e] += b.get(e);
                    }
                }
            }
        };
        const uint32_t acc_empty_lead = CL > 1 ? mapa_shared(acc_empty, 0) : 0;
        if constexpr (AUX_IN)
            for (int g = 0; g < AHEAD; g++) aux_issue(g);
        for (int u = ufirst; u < units && alive; u += ustep, local++) {
            int sp, mt, nt, lb;
            decode(u, sp, mt, nt, lb);
            const int acc = local % NACC;
            const uint32_t aph = (local / NACC) & 1;
            // one lane waits; the warp then proceeds converged (tcgen05.ld is warp-wide)
            int okw = 1;
            if (lane == 0) okw = mbar_wait(&acc_full[acc], aph, abort_flag, err) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (!okw) break;
            __syncwarp();
            tc_fence_after();
            const int row0 = mt * TC_BM + lane_grp * 32;   // first of this warp's 32 rows
            const int oy = lb * ep.o_rows;                 // batch element's first output row
            const int yout = ((EPI == TC_EPI_PARTIAL) ? sp * M + row0 : row0) + oy;
#pragma unroll 1
            for (int pi = 0; pi < NPAIR && alive; pi++) {
                const int c = cbase + pi * 64;
                if (!AUX_IN && nt * BN + c >= N) break;
                uint32_t r0[32], r1[32];
                const uint32_t ta = tmem_base + ((uint32_t)(lane_grp * 32) << 16) + acc * BN + c;
                tmem_ld32(ta, r0);
                tmem_ld32(ta + 32, r1);
                tmem_ld_wait();
                float v2[64];
#pragma unroll
                for (int i = 0; i < 32; i++) { v2[i] = __uint_as_float(r0[i]); v2[32 + i] = __uint_as_float(r1[i]); }
                if constexpr (F8) {
                    // unscale: this lane's row factor times the weight's factor
                    const int row = row0 + lane;
                    const float sc = (row < M ? ep.a_deq[row] : 0.f) * ep.b_deq[0];
#pragma unroll
                    for (int i = 0; i < 64; i++) v2[i] *= sc;
                }
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    float* v = v2 + 32 * h;
                    const int col = nt * BN + c + 32 * h;      // first global column of the piece
                    if constexpr (EPI == EPI_ACC_F32 || EPI == TC_EPI_PARTIAL) {
                        if (col < N) {
#pragma unroll
                            for (int q = 0; q < 2; q++) {          // 16 fp32 columns per 64-byte row
                                uint8_t* sb = stg + (nbuf % NB) * S::STG_BYTES;
                                if (lane == 0) bulk_wait_read<NB - 1>();
                                __syncwarp();
#pragma unroll
                                for (int j = 0; j < 4; j++)
                                    *reinterpret_cast<float4*>(sb + stg_off(lane, j)) =
                                        make_float4(v[16 * q + 4 * j], v[16 * q + 4 * j + 1], v[16 * q + 4 * j + 2],
                                                    v[16 * q + 4 * j + 3]);
                                fence_async_smem();
                                __syncwarp();
                                if (lane == 0 && col + 16 * q < N) {
                                    if constexpr (EPI == EPI_ACC_F32) tma_reduce_add_2d(&tmOut, sb, col + 16 * q, yout);
                                    else tma_store_2d(&tmOut, sb, col + 16 * q, yout);
                                    bulk_commit();
                                }
                                nbuf++;
                            }
                        }
                    } else if constexpr (AUX_IN) {
                        // this piece's input was loaded into buffer nbuf % NB ahead of time
                        // (nbuf counts this warp's pieces); start the load AHEAD pieces on
                        const int kb = nbuf % NB;
                        aux_issue(nbuf + AHEAD);
                        int oka = 1;
                        if (lane == 0) oka = mbar_wait(&auxb[kb], (aux_ph >> kb) & 1, abort_flag, err) ? 1 : 0;
                        oka = __shfl_sync(0xffffffffu, oka, 0);
                        aux_ph ^= 1u << kb;
                        aux_pend &= ~(1u << kb);
                        if (!oka) { alive = false; break; }
                        __syncwarp();
                        uint8_t* sb = stg + kb * S::STG_BYTES;
                        if (EPI == EPI_RESID) add_bias(v, col);
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            Vec<bf16> a, o;
                            a.v = *reinterpret_cast<const uint4*>(sb + stg_off(lane, j));
#pragma unroll
                            for (int e = 0; e < 8; e += 2) {
                                const float2 x = a.get2(e), acc2 = make_float2(v[8 * j + e], v[8 * j + e + 1]);
                                const float2 r = (EPI == EPI_RESID) ? __fadd2_rn(acc2, x)
                                                 : __fmul2_rn(acc2, ep.gelu_deriv ? x : gelu_grad2_fast(x));
                                o.set2(e, r.x, r.y);
                            }
                            *reinterpret_cast<uint4*>(sb + stg_off(lane, j)) = o.v;
                        }
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0 && col < N) { tma_store_2d(&tmOut, sb, col, yout); bulk_commit(); }
                        nbuf++;
                        if (EPI == EPI_GELU_BWD && ep.csum) {
                            // the bias gradient of the layer whose pre-activation this is:
                            // this piece's 32 column sums over the warp's 32 rows, read
                            // back from the staged (stored) values.  Lane: column pair
                            // lane % 16 of the even (lane < 16) or odd rows
                            const int cp = lane & 15, odd = lane >> 4;
                            const int nrow = M - row0;
                            float2 p[16];
#pragma unroll
                            for (int k = 0; k < 16; k++) {
                                const int rr = 2 * k + odd;
                                const uint32_t u = *reinterpret_cast<const uint32_t*>(sb + stg_off(rr, cp >> 2) + (cp & 3) * 4);
                                p[k] = rr < nrow ? make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u))
                                                 : make_float2(0.f, 0.f);
                            }
#pragma unroll
                            for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                                for (int k = 0; k < w; k++) p[k] = __fadd2_rn(p[k], p[k + w]);
                            float2 acc2 = p[0];
                            acc2.x += __shfl_xor_sync(0xffffffffu, acc2.x, 16);
                            acc2.y += __shfl_xor_sync(0xffffffffu, acc2.y, 16);
                            if (!odd && col + 2 * cp < N)
                                *reinterpret_cast<float2*>(ep.csum + (size_t)(row0 >> 5) * N + col + 2 * cp) = acc2;
                        }
                    } else {
                        if (col < N) {
                            add_bias(v, col);
                            uint8_t* sb = stg + (nbuf % NB) * S::STG_BYTES;
                            if (lane == 0) bulk_wait_read<NB - 1>();
                            __syncwarp();
                            if constexpr (EPI == EPI_GELU) {
                                // pre-activation (or its GELU derivative) out first, then the
                                // activation into the other buffer; both of the rounded (bf16)
                                // pre-activation
#pragma unroll
                                for (int j = 0; j < 4; j++) {
                                    Vec<bf16> o;
#pragma unroll
                                    for (int e = 0; e < 8; e += 2) o.set2(e, v[8 * j + e], v[8 * j + e + 1]);
                                    if (ep.gelu_deriv) {
                                        Vec<bf16> dv;
#pragma unroll
                                        for (int e = 0; e < 8; e += 2) {
                                            float2 g, d;
                                            gelu_and_grad2_fast(o.get2(e), g, d);
                                            v[8 * j + e] = g.x;
                                            v[8 * j + e + 1] = g.y;
                                            dv.set2(e, d.x, d.y);
                                        }
                                        *reinterpret_cast<uint4*>(sb + stg_off(lane, j)) = dv.v;
                                    } else {
                                        *reinterpret_cast<uint4*>(sb + stg_off(lane, j)) = o.v;
#pragma unroll
                                        for (int e = 0; e < 8; e += 2) {
                                            const float2 g = gelu2_fast(o.get2(e));      // of the stored pre-activation
                                            v[8 * j + e] = g.x;
                                            v[8 * j + e + 1] = g.y;
                                        }
                                    }
                                }
                                fence_async_smem();
                                __syncwarp();
                                if (lane == 0) { tma_store_2d(&tmAux, sb, col, row0 + oy); bulk_commit(); }
                                nbuf++;
                                sb = stg + (nbuf % NB) * S::STG_BYTES;
                                if (lane == 0) bulk_wait_read<NB - 1>();
                                __syncwarp();
                            }
#pragma unroll
                            for (int j = 0; j < 4; j++) {
                                Vec<bf16> o;
#pragma unroll
                                for (int e = 0; e < 8; e += 2) o.set2(e, v[8 * j + e], v[8 * j + e + 1]);
                                *reinterpret_cast<uint4*>(sb + stg_off(lane, j)) = o.v;
                            }
                            fence_async_smem();
                            __syncwarp();
                            if (lane == 0) { tma_store_2d(&tmOut, sb, col, yout); bulk_commit(); }
                            nbuf++;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (CL == 1 || leader) mbar_arrive(&acc_empty[acc]);
                else mbar_arrive_cluster(acc_empty_lead + acc * 8);     // the pair's accumulator lives on
            }
        }
        // every store this warp issued has completed, and no load is still landing in
        // its staging buffers (only possible after an abort), before the CTA retires
        if (lane == 0) {
            bulk_wait<0>();
            for (int kb = 0; kb < NB; kb++) {
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
    // the peer's multicast commits to this CTA's barriers have all landed (its MMA thread
    // waited for its own MMAs) before either CTA of the cluster exits
    if (CL > 1) cluster_sync();
    tc_fence_after();
    __syncwarp();
    if (warp == 1) {
        if constexpr (CL == 1)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(NACC * BN)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(NACC * BN)
                         : "memory");
    }
}

// out[n][k] += sum_s part[s][n][k], s in order (split-K reduction, deterministic; with
// `assign`, out = 0 + the same sum).  All
// of a packet's partial loads (splits <= TC_MAX_SPLITS) are issued before the first add.
#define TC_MAX_SPLITS 8
__global__ void splitk_reduce_kernel(float* __restrict__ out, const float* __restrict__ part, size_t n4,
                                     int splits, int assign) {
    pdl_wait();
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 p[TC_MAX_SPLITS];
#pragma unroll
    for (int s = 0; s < TC_MAX_SPLITS; s++)
        if (s < splits) p[s] = __ldcs(reinterpret_cast<const float4*>(part) + (size_t)s * n4 + i);
    // assign: the output's first write of the step (0 + the partials, in the same order)
    float4 acc = assign ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<float4*>(out)[i];
#pragma unroll
    for (int s = 0; s < TC_MAX_SPLITS; s++) {
        if (s < splits) { acc.x += p[s].x; acc.y += p[s].y; acc.z += p[s].z; acc.w += p[s].w; }
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
// SMs, with at most TC_MAX_SPLITS splits: its partials never exceed 8 x (SMs x one tile).
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
    const CUtensorMapDataType dt = ebytes == 2   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : ebytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// epilogue map: box of 64-byte rows x 32 rows (32 bf16 or 16 fp32 columns), 64-byte
// swizzle, matching the epilogue's 2 KB staging buffers
static bool make_epi_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                         int ebytes = 2) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * ebytes};
    cuuint32_t box[2] = {(cuuint32_t)(64 / ebytes), 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, ebytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

template <int BN, int EPI, bool A_MN, bool B_MN, int CL = 1, bool F8 = false>
static int launch_tc(cudaStream_t s, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to,
                     const CUtensorMap& tx, int M, int N, int K, int splits, const TcEpi& ep, unsigned* err) {
    using SM = TcSmem<BN, CL, TcBufs<EPI, CL>::value>;
    static int max_clusters = 0;            // co-resident clusters of CL CTAs (0: not yet queried)
    auto kern = gemm_tc_kernel<BN, EPI, A_MN, B_MN, CL, F8>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = SM::TOTAL;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;    // see launch_pdl
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_clusters == 0) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::TOTAL) != cudaSuccess)
            return GPT2_ECUDA;
        cfg.gridDim = dim3(g_num_sms / CL * CL);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) return GPT2_ECUDA;
        max_clusters = n;
    }
    const int units = ((M + TC_BM - 1) / TC_BM + CL - 1) / CL * ((N + BN - 1) / BN) * splits * (ep.nb > 1 ? ep.nb : 1);
    const int clusters = units < max_clusters ? units : max_clusters;
    cfg.gridDim = dim3(clusters * CL);
    cfg.numAttrs = 2;
    // stream the larger operand once: m fastest when B (N x K) is larger than A (M x K)
    const int m_fast = N > M ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, to, tx, M, N, K, splits, m_fast, ep, err) != cudaSuccess)
        return GPT2_ECUDA;
    rt_note_launches(1);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}

int gemm_tc_forward(cudaStream_t s, bf16* out, const bf16* inp, const bf16* W, const bf16* bias, int M, int N,
                    int K, int epi, bf16* aux, unsigned* err, bool gelu_deriv) {
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (N % 8 || K % 8 || M < 1 || !aligned16(out) || !aligned16(inp) || !aligned16(W) ||
        (bias && !aligned16(bias)) || (aux && !aligned16(aux)))
        return GPT2_EUNSUPPORTED;
    CUtensorMap ta, tb, to, tx;
    // CTA pairs (256 x 256 tiles, half of B per CTA) except for the smallest products,
    // where the halved unit count costs more than the pair saves
    const int cl = (N <= 768 && K <= 768) ? 1 : 2;
    if (!make_map(&ta, inp, K, M, K, TC_BM) || !make_map(&tb, W, K, N, K, 256 / cl) ||
        !make_epi_map(&to, out, N, M, N))
        return GPT2_EUNSUPPORTED;
    if (aux) {
        if (!make_epi_map(&tx, aux, N, M, N)) return GPT2_EUNSUPPORTED;
    } else {
        tx = to;
    }
    TcEpi ep{out, bias, aux, (long)N};
    ep.gelu_deriv = gelu_deriv ? 1 : 0;
    switch (epi) {
        case EPI_STORE:
            return cl == 2 ? launch_tc<256, EPI_STORE, false, false, 2>(s, ta, tb, to, tx, M, N, K, 1, ep, err)
                           : launch_tc<256, EPI_STORE, false, false, 1>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        case EPI_GELU:
            return cl == 2 ? launch_tc<256, EPI_GELU, false, false, 2>(s, ta, tb, to, tx, M, N, K, 1, ep, err)
                           : launch_tc<256, EPI_GELU, false, false, 1>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        case EPI_RESID:
            return cl == 2 ? launch_tc<256, EPI_RESID, false, false, 2>(s, ta, tb, to, tx, M, N, K, 1, ep, err)
                           : launch_tc<256, EPI_RESID, false, false, 1>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        default: return GPT2_EUNSUPPORTED;
    }
}

int gemm_tc_forward_fp8(cudaStream_t s, bf16* out, const uint8_t* inp, const float* inp_deq, const uint8_t* W,
                        const float* w_deq, const bf16* bias, int M, int N, int K, int epi, bf16* aux, unsigned* err,
                        bool gelu_deriv) {
    // as gemm_tc_forward with e4m3 operands: K a multiple of 16 (16-byte rows for TMA)
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (N % 8 || K % 16 || M < 1 || !inp_deq || !w_deq || !aligned16(out) || !aligned16(inp) || !aligned16(W) ||
        (bias && !aligned16(bias)) || (aux && !aligned16(aux)))
        return GPT2_EUNSUPPORTED;
    CUtensorMap ta, tb, to, tx;
    const int cl = (N <= 768 && K <= 768) ? 1 : 2;
    if (!make_map(&ta, inp, K, M, K, TC_BM, 1) || !make_map(&tb, W, K, N, K, 256 / cl, 1) ||
        !make_epi_map(&to, out, N, M, N))
        return GPT2_EUNSUPPORTED;
    if (aux) {
        if (!make_epi_map(&tx, aux, N, M, N)) return GPT2_EUNSUPPORTED;
    } else {
        tx = to;
    }
    TcEpi ep{out, bias, aux, (long)N, inp_deq, w_deq};
    ep.gelu_deriv = gelu_deriv ? 1 : 0;
    switch (epi) {
        case EPI_STORE:
            return cl == 2 ? launch_tc<256, EPI_STORE, false, false, 2, true>(s, ta, tb, to, tx, M, N, K, 1, ep, err)
                           : launch_tc<256, EPI_STORE, false, false, 1, true>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        case EPI_GELU:
            return cl == 2 ? launch_tc<256, EPI_GELU, false, false, 2, true>(s, ta, tb, to, tx, M, N, K, 1, ep, err)
                           : launch_tc<256, EPI_GELU, false, false, 1, true>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        case EPI_RESID:
            return cl == 2 ? launch_tc<256, EPI_RESID, false, false, 2, true>(s, ta, tb, to, tx, M, N, K, 1, ep, err)
                           : launch_tc<256, EPI_RESID, false, false, 1, true>(s, ta, tb, to, tx, M, N, K, 1, ep, err);
        default: return GPT2_EUNSUPPORTED;
    }
}

int gemm_tc_bf16_batched(cudaStream_t s, bf16* out, const bf16* A, bool a_mn, const bf16* B, bool b_mn, int M, int N,
                         int K, int nb, unsigned* err) {
    // out_l (M x N) = sum_k A_l(m,k) B_l(n,k), l < nb, each operand's nb matrices
    // contiguous: A K-major (M rows of K) or MN-major (K rows of M), B K-major (N rows of K)
    // or MN-major (K rows of N).  In the tensor maps the matrices are stacked along their
    // rows, so with nb > 1 no tile may straddle two of them: M, N multiples of 256, K of 64.
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (M % 8 || N % 8 || K % 8 || nb < 1 || !aligned16(out) || !aligned16(A) || !aligned16(B))
        return GPT2_EUNSUPPORTED;
    if (nb > 1 && (M % 256 || N % 256 || K % 64)) return GPT2_EUNSUPPORTED;
    const int cl = (N <= 768 && K <= 768) ? 1 : 2;
    CUtensorMap ta, tb, to;
    const uint64_t nbu = (uint64_t)nb;
    const bool ok_a = a_mn ? make_map(&ta, A, M, K * nbu, M, 64) : make_map(&ta, A, K, M * nbu, K, TC_BM);
    const bool ok_b = b_mn ? make_map(&tb, B, N, K * nbu, N, 64) : make_map(&tb, B, K, N * nbu, K, 256 / cl);
    if (!ok_a || !ok_b || !make_epi_map(&to, out, N, M * nbu, N)) return GPT2_EUNSUPPORTED;
    TcEpi ep{out, nullptr, nullptr, (long)N};
    ep.nb = nb;
    ep.a_rows = a_mn ? K : M;
    ep.b_rows = b_mn ? K : N;
    ep.o_rows = M;
    if (!a_mn && !b_mn)
        return cl == 2 ? launch_tc<256, EPI_STORE, false, false, 2>(s, ta, tb, to, to, M, N, K, 1, ep, err)
                       : launch_tc<256, EPI_STORE, false, false, 1>(s, ta, tb, to, to, M, N, K, 1, ep, err);
    if (!a_mn && b_mn)
        return cl == 2 ? launch_tc<256, EPI_STORE, false, true, 2>(s, ta, tb, to, to, M, N, K, 1, ep, err)
                       : launch_tc<256, EPI_STORE, false, true, 1>(s, ta, tb, to, to, M, N, K, 1, ep, err);
    if (a_mn && b_mn)
        return cl == 2 ? launch_tc<256, EPI_STORE, true, true, 2>(s, ta, tb, to, to, M, N, K, 1, ep, err)
                       : launch_tc<256, EPI_STORE, true, true, 1>(s, ta, tb, to, to, M, N, K, 1, ep, err);
    return GPT2_EUNSUPPORTED;
}

int gemm_tc_bf16(cudaStream_t s, bf16* out, const bf16* A, bool a_mn, const bf16* B, bool b_mn, int M, int N, int K,
                 unsigned* err) {
    return gemm_tc_bf16_batched(s, out, A, a_mn, B, b_mn, M, N, K, 1, err);
}

int gemm_tc_backward_dx(cudaStream_t s, bf16* dinp, const bf16* dout, const bf16* W, int M, int N, int K, int epi,
                        const bf16* aux, float* csum, unsigned* err, bool gelu_deriv) {
    // dinp (M x K) = dout (M x N) W (N x K): contraction over N; A = dout K-major,
    // B(k_out, n) = W[n][k_out] is MN-major (k_out contiguous)
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (N % 8 || K % 8 || M < 1 || !aligned16(dinp) || !aligned16(dout) || !aligned16(W) ||
        (aux && !aligned16(aux)))
        return GPT2_EUNSUPPORTED;
    CUtensorMap ta, tb, to, tx;
    if (!make_map(&ta, dout, N, M, N, TC_BM) || !make_map(&tb, W, K, N, K, 64) || !make_epi_map(&to, dinp, K, M, K))
        return GPT2_EUNSUPPORTED;
    if (aux) {
        if (!make_epi_map(&tx, aux, K, M, K)) return GPT2_EUNSUPPORTED;
    } else {
        tx = to;
    }
    if (csum && epi != EPI_GELU_BWD) return GPT2_EINVAL;
    TcEpi ep{dinp, nullptr, (void*)aux, (long)K, nullptr, nullptr, csum};
    ep.gelu_deriv = gelu_deriv ? 1 : 0;
    const int cl = (N <= 768 && K <= 768) ? 1 : 2;      // as in the forward
    if (epi == EPI_GELU_BWD)
        return cl == 2 ? launch_tc<256, EPI_GELU_BWD, false, true, 2>(s, ta, tb, to, tx, M, K, N, 1, ep, err)
                       : launch_tc<256, EPI_GELU_BWD, false, true, 1>(s, ta, tb, to, tx, M, K, N, 1, ep, err);
    if (epi == EPI_STORE)
        return cl == 2 ? launch_tc<256, EPI_STORE, false, true, 2>(s, ta, tb, to, tx, M, K, N, 1, ep, err)
                       : launch_tc<256, EPI_STORE, false, true, 1>(s, ta, tb, to, tx, M, K, N, 1, ep, err);
    return GPT2_EUNSUPPORTED;
}

static int choose_splits(int tiles, int nkb, int slots) {
    // with fewer tiles than slots (SMs, or CTA pairs), fill them: the split count with
    // the best occupancy over whole waves, each split keeping at least 8 k-blocks
    if (tiles >= slots || g_num_sms > TC_SPLIT_SM_BOUND) return 1;
    int best = 1;
    double best_eff = 0;
    for (int sp = 1; sp <= TC_MAX_SPLITS; sp++) {
        if (sp > 1 && nkb / sp < 8) break;
        const int units = tiles * sp;
        const int waves = (units + slots - 1) / slots;
        const double eff = (double)units / (waves * slots);
        if (eff > best_eff + 1e-9) { best_eff = eff; best = sp; }
    }
    return best;
}

int gemm_tc_backward_dw(cudaStream_t s, float* dW, const bf16* dout, const bf16* inp, int M, int N, int K,
                        float* scratch, size_t scratch_floats, unsigned* err, bool assign) {
    // dW (N x K) += dout^T (N x M) inp (M x K): contraction over M; A(n, m) = dout[m][n]
    // and B(k, m) = inp[m][k] are both MN-major
    if (!gemm_tc_available()) return GPT2_EUNSUPPORTED;
    if (N % 8 || K % 8 || M < 1 || !aligned16(dW) || !aligned16(dout) || !aligned16(inp))
        return GPT2_EUNSUPPORTED;
    CUtensorMap ta, tb, to;
    if (!make_map(&ta, dout, N, M, N, 64) || !make_map(&tb, inp, K, M, K, 64)) return GPT2_EUNSUPPORTED;
    // 256-wide tiles throughout (measured faster than 128-wide tiles for every weight
    // gradient of the model), on CTA pairs (256 x 256 tiles) when the 256-row groups tile
    // N exactly; split-K fills the GPU when there are fewer tiles than SMs (pairs)
    const bool okpair = N % (2 * TC_BM) == 0;
    const int cl = okpair ? 2 : 1;
    const int tiles = ((N + cl * TC_BM - 1) / (cl * TC_BM)) * ((K + 255) / 256);
    const int nkb = (M + TC_BK - 1) / TC_BK;
    int splits = choose_splits(tiles, nkb, g_num_sms / cl);
    // partial tiles of split s are rows [s*N, (s+1)*N) of one map, so a tile (pair) must
    // not straddle two splits: N a multiple of the tile (pair) height
    if (splits > 1 && (!scratch || (size_t)splits * N * K > scratch_floats || !aligned16(scratch) || N % (cl * TC_BM)))
        splits = 1;
    if (splits == 1) {
        if (!make_epi_map(&to, dW, K, N, K, 4)) return GPT2_EUNSUPPORTED;
        TcEpi ep{dW, nullptr, nullptr, (long)K};
        // assign: the tile is stored (the partial-tile epilogue with one split) instead of
        // added by a TMA reduction -- the same values as adding into zeros
        if (assign)
            return cl == 2 ? launch_tc<256, TC_EPI_PARTIAL, true, true, 2>(s, ta, tb, to, to, N, K, M, 1, ep, err)
                           : launch_tc<256, TC_EPI_PARTIAL, true, true, 1>(s, ta, tb, to, to, N, K, M, 1, ep, err);
        return cl == 2 ? launch_tc<256, EPI_ACC_F32, true, true, 2>(s, ta, tb, to, to, N, K, M, 1, ep, err)
                       : launch_tc<256, EPI_ACC_F32, true, true, 1>(s, ta, tb, to, to, N, K, M, 1, ep, err);
    }
    if (!make_epi_map(&to, scratch, K, (uint64_t)splits * N, K, 4)) return GPT2_EUNSUPPORTED;
    TcEpi ep{scratch, nullptr, nullptr, (long)K};
    int rc = cl == 2 ? launch_tc<256, TC_EPI_PARTIAL, true, true, 2>(s, ta, tb, to, to, N, K, M, splits, ep, err)
                     : launch_tc<256, TC_EPI_PARTIAL, true, true, 1>(s, ta, tb, to, to, N, K, M, splits, ep, err);
    if (rc != GPT2_OK) return rc;
    const size_t n4 = (size_t)N * K / 4;
    launch_pdl(splitk_reduce_kernel, (unsigned)((n4 + 255) / 256), 256, 0, s, dW, scratch, n4, splits, assign ? 1 : 0);
    rt_note_launches(1);
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ECUDA;
}
