// Tensor-core (mma.sync m16n8k16, bf16 -> fp32) flash attention for head size 64.
//
// ujoy.net llm.c article, section "用C语言实现LLM": causal self-attention forward and
// backward.  Per head: S = Q K^T / sqrt(64) over keys j <= t, P = softmax(S), O = P V;
// backward with D = rowsum(dO * O): dV = P^T dO, dP = dO V^T, dS = P (dP - D),
// dQ = dS K / 8, dK = dS^T Q / 8.
//
// Forward: a CTA takes 128 queries of one (b, h) (8 warps x 16 rows) and streams
// 64-key blocks of K and V through shared memory (cp.async, double-buffered), keeping
// an online softmax in registers; only O and the row log-sum-exp are written.
// Backward, without atomics: one kernel per 64-key block accumulates dK, dV over the
// query blocks at or after it; another per 64-query block accumulates dQ over the key
// blocks up to the diagonal.  P is recomputed from Q, K and the saved LSE.
//
// Shared-memory tiles are 64 bf16 (128 bytes) per row with the 16-byte chunk index
// XOR-ed by (row % 8), so the 8 row addresses of every ldmatrix hit distinct banks.
#pragma once
#include "common.cuh"

#define AM_HS 64
#define AM_LOG2E 1.4426950408889634f

__device__ __forceinline__ uint32_t am_smem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// element offset of (row, 16-byte chunk) in a swizzled 64-wide tile
__device__ __forceinline__ int am_sw(int row, int chunk) { return row * AM_HS + ((chunk ^ (row & 7)) << 3); }

__device__ __forceinline__ void am_cp16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(am_smem(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void am_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void am_cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void am_ldsm4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(am_smem(p)));
}
__device__ __forceinline__ void am_ldsm4t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(am_smem(p)));
}
__device__ __forceinline__ void am_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t am_pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Copy `rows` rows (64 bf16 each, row pitch `ld` elements, starting at row r0 of a
// sequence of length Tn) into a swizzled tile; rows >= Tn are zero-filled.
template <int ROWS, int NTHREADS>
__device__ __forceinline__ void am_load_tile(bf16* tile, const bf16* base, long ld, int r0, int Tn) {
#pragma unroll
    for (int i = threadIdx.x; i < ROWS * 8; i += NTHREADS) {
        const int r = i >> 3, c = i & 7;
        const bool ok = (r0 + r) < Tn;
        const bf16* src = base + (size_t)(ok ? (r0 + r) : 0) * ld + c * 8;
        am_cp16(tile + am_sw(r, c), src, ok);
    }
}

// A fragments (16 rows x 64 columns, 4 k-steps) of rows [row0, row0+16) of a tile
__device__ __forceinline__ void am_load_afrag(uint32_t (&a)[4][4], const bf16* tile, int row0) {
    const int l = threadIdx.x & 31, mi = l >> 3;
#pragma unroll
    for (int s = 0; s < 4; s++) am_ldsm4(a[s], tile + am_sw(row0 + (mi & 1) * 8 + (l & 7), 2 * s + (mi >> 1)));
}

// acc[16 x 64] (8 n8-tiles) += A (16 x 64, fragments) * B, with B(k, n) = tile[n][k]
// (rows of the tile are the n index): non-transposed ldmatrix of tile rows.
__device__ __forceinline__ void am_mm_rows(float (&acc)[8][4], const uint32_t (&a)[4][4], const bf16* tile) {
    const int l = threadIdx.x & 31, mi = l >> 3;
#pragma unroll
    for (int s = 0; s < 4; s++) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            uint32_t b[4];
            am_ldsm4(b, tile + am_sw(j * 8 + (mi >> 1) * 8 + (l & 7), 2 * s + (mi & 1)));
            am_mma(acc[j], a[s], b[0], b[1]);
            am_mma(acc[j + 1], a[s], b[2], b[3]);
        }
    }
}

// acc[16 x 64] += A (16 x 64 over the tile's rows as k) * tile, B(k, n) = tile[k][n]:
// transposed ldmatrix.
__device__ __forceinline__ void am_mm_cols(float (&acc)[8][4], const uint32_t (&a)[4][4], const bf16* tile) {
    const int l = threadIdx.x & 31, mi = l >> 3;
#pragma unroll
    for (int s = 0; s < 4; s++) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            uint32_t b[4];
            am_ldsm4t(b, tile + am_sw(16 * s + (mi & 1) * 8 + (l & 7), j + (mi >> 1)));
            am_mma(acc[j], a[s], b[0], b[1]);
            am_mma(acc[j + 1], a[s], b[2], b[3]);
        }
    }
}

// Accumulators of a 16 x 64 product as bf16 A fragments (4 k-steps of 16 columns).
__device__ __forceinline__ void am_acc_to_afrag(uint32_t (&a)[4][4], const float (&c)[8][4]) {
#pragma unroll
    for (int s = 0; s < 4; s++) {
        a[s][0] = am_pack(c[2 * s][0], c[2 * s][1]);
        a[s][1] = am_pack(c[2 * s][2], c[2 * s][3]);
        a[s][2] = am_pack(c[2 * s + 1][0], c[2 * s + 1][1]);
        a[s][3] = am_pack(c[2 * s + 1][2], c[2 * s + 1][3]);
    }
}

// ============================================================== forward
#define AMF_Q 128
#define AMF_K 64
#define AMF_THREADS 256
__global__ void __launch_bounds__(AMF_THREADS)
attention_forward_mma(bf16* __restrict__ out, float* __restrict__ lse, const bf16* __restrict__ qkv,
                      int B, int Tn, int C, int NH) {
    __shared__ __align__(128) bf16 Qs[AMF_Q * AM_HS];
    __shared__ __align__(128) bf16 Ks[2][AMF_K * AM_HS];
    __shared__ __align__(128) bf16 Vs[2][AMF_K * AM_HS];
    const int nqb = (Tn + AMF_Q - 1) / AMF_Q;
    const int qb = nqb - 1 - blockIdx.x;          // longest rows first
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int C3 = 3 * C;
    const bf16* base = qkv + (size_t)b * Tn * C3;
    const bf16* qg = base + h * AM_HS;
    const bf16* kg = base + C + h * AM_HS;
    const bf16* vg = base + 2 * C + h * AM_HS;
    const int warp = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
    const int q0 = qb * AMF_Q;
    const int wq0 = q0 + warp * 16;                // this warp's first query row
    const int nkb = min((Tn + AMF_K - 1) / AMF_K, (q0 + AMF_Q - 1) / AMF_K + 1);

    am_load_tile<AMF_Q, AMF_THREADS>(Qs, qg, C3, q0, Tn);
    am_load_tile<AMF_K, AMF_THREADS>(Ks[0], kg, C3, 0, Tn);
    am_load_tile<AMF_K, AMF_THREADS>(Vs[0], vg, C3, 0, Tn);
    am_cp_commit();

    const float sl2 = AM_LOG2E / 8.0f;             // 1/sqrt(64) in the exp2 domain
    float m[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
    float o[8][4];
#pragma unroll
    for (int j = 0; j < 8; j++) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    uint32_t qa[4][4];

    for (int kb = 0; kb < nkb; kb++) {
        const int buf = kb & 1;
        if (kb + 1 < nkb) {
            am_load_tile<AMF_K, AMF_THREADS>(Ks[buf ^ 1], kg, C3, (kb + 1) * AMF_K, Tn);
            am_load_tile<AMF_K, AMF_THREADS>(Vs[buf ^ 1], vg, C3, (kb + 1) * AMF_K, Tn);
        }
        am_cp_commit();
        am_cp_wait<1>();
        __syncthreads();
        if (kb == 0) am_load_afrag(qa, Qs, warp * 16);
        const int k0 = kb * AMF_K;
        if (k0 <= wq0 + 15) {                       // some key of this block is visible to the warp
            float s[8][4];
#pragma unroll
            for (int j = 0; j < 8; j++) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
            am_mm_rows(s, qa, Ks[buf]);
            const bool diag = k0 + AMF_K - 1 > wq0;
#pragma unroll
            for (int j = 0; j < 8; j++)
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    float x = s[j][e] * sl2;
                    if (diag) {
                        const int key = k0 + j * 8 + 2 * t + (e & 1);
                        const int q = wq0 + g + (e >> 1) * 8;
                        if (key > q) x = -INFINITY;
                    }
                    s[j][e] = x;
                }
#pragma unroll
            for (int r = 0; r < 2; r++) {
                float mx = m[r];
#pragma unroll
                for (int j = 0; j < 8; j++) mx = fmaxf(mx, fmaxf(s[j][2 * r], s[j][2 * r + 1]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float corr = exp2f(m[r] - mx);
                m[r] = mx;
                float rs = 0.f;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    s[j][2 * r] = exp2f(s[j][2 * r] - mx);
                    s[j][2 * r + 1] = exp2f(s[j][2 * r + 1] - mx);
                    rs += s[j][2 * r] + s[j][2 * r + 1];
                }
                lsum[r] = lsum[r] * corr + rs;
#pragma unroll
                for (int j = 0; j < 8; j++) { o[j][2 * r] *= corr; o[j][2 * r + 1] *= corr; }
            }
            uint32_t pa[4][4];
            am_acc_to_afrag(pa, s);
            am_mm_cols(o, pa, Vs[buf]);
        }
        __syncthreads();
    }
    // row sums are spread over the 4 threads of a quad
#pragma unroll
    for (int r = 0; r < 2; r++) {
        lsum[r] += __shfl_xor_sync(0xffffffffu, lsum[r], 1);
        lsum[r] += __shfl_xor_sync(0xffffffffu, lsum[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int q = wq0 + g + r * 8;
        if (q >= Tn) continue;
        const float inv = 1.0f / lsum[r];
        bf16* orow = out + ((size_t)b * Tn + q) * C + h * AM_HS;
#pragma unroll
        for (int j = 0; j < 8; j++)
            *reinterpret_cast<uint32_t*>(orow + j * 8 + 2 * t) = am_pack(o[j][2 * r] * inv, o[j][2 * r + 1] * inv);
        if (t == 0) lse[((size_t)b * NH + h) * Tn + q] = (m[r] + log2f(lsum[r])) / AM_LOG2E;
    }
}

// ============================================================== backward: dK, dV
#define AMB_ROWS 64
#define AMB_THREADS 128
__global__ void __launch_bounds__(AMB_THREADS)
attention_backward_dkv_mma(bf16* __restrict__ dqkv, const bf16* __restrict__ dout, const bf16* __restrict__ qkv,
                           const float* __restrict__ lse, const float* __restrict__ Dsum, int B, int Tn, int C,
                           int NH) {
    __shared__ __align__(128) bf16 Ks[AMB_ROWS * AM_HS];
    __shared__ __align__(128) bf16 Vs[AMB_ROWS * AM_HS];
    __shared__ __align__(128) bf16 Qs[2][AMB_ROWS * AM_HS];
    __shared__ __align__(128) bf16 dOs[2][AMB_ROWS * AM_HS];
    const int nb = (Tn + AMB_ROWS - 1) / AMB_ROWS;
    const int kbk = blockIdx.x;                   // key block (block 0 has the most work; it starts first)
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int C3 = 3 * C;
    const bf16* base = qkv + (size_t)b * Tn * C3;
    const bf16* qg = base + h * AM_HS;
    const bf16* kg = base + C + h * AM_HS;
    const bf16* vg = base + 2 * C + h * AM_HS;
    const bf16* dog = dout + (size_t)b * Tn * C + h * AM_HS;
    const float* lg = lse + (size_t)bh * Tn;
    const float* dg = Dsum + (size_t)bh * Tn;
    const int warp = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
    const int k0 = kbk * AMB_ROWS;
    const int wk0 = k0 + warp * 16;                // this warp's first key

    auto load_q = [&](int qbi, int buf) {
        am_load_tile<AMB_ROWS, AMB_THREADS>(Qs[buf], qg, C3, qbi * AMB_ROWS, Tn);
        am_load_tile<AMB_ROWS, AMB_THREADS>(dOs[buf], dog, C, qbi * AMB_ROWS, Tn);
    };
    am_load_tile<AMB_ROWS, AMB_THREADS>(Ks, kg, C3, k0, Tn);
    am_load_tile<AMB_ROWS, AMB_THREADS>(Vs, vg, C3, k0, Tn);
    load_q(kbk, 0);
    am_cp_commit();

    const float sl2 = AM_LOG2E / 8.0f;
    uint32_t ka[4][4], va[4][4];
    float dk[8][4], dv[8][4];
#pragma unroll
    for (int j = 0; j < 8; j++)
#pragma unroll
        for (int e = 0; e < 4; e++) { dk[j][e] = 0.f; dv[j][e] = 0.f; }

    for (int qbi = kbk; qbi < nb; qbi++) {
        const int buf = (qbi - kbk) & 1;
        if (qbi + 1 < nb) {
            __syncthreads();                        // the other buffer's last readers are done
            load_q(qbi + 1, buf ^ 1);
        }
        am_cp_commit();
        am_cp_wait<1>();
        __syncthreads();
        if (qbi == kbk) {
            am_load_afrag(ka, Ks, warp * 16);
            am_load_afrag(va, Vs, warp * 16);
        }
        const int q0 = qbi * AMB_ROWS;
        if (q0 + AMB_ROWS - 1 < wk0) continue;     // every query of the block precedes this warp's keys
        // LSE (exp2 domain) and D of the 16 query columns this thread holds
        float Lq[8][2], Dq[8][2];
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int c = 0; c < 2; c++) {
                const int q = q0 + j * 8 + 2 * t + c;
                Lq[j][c] = q < Tn ? __ldg(lg + q) * AM_LOG2E : 0.f;
                Dq[j][c] = q < Tn ? __ldg(dg + q) : 0.f;
            }
        // S^T (16 keys x 64 queries) and dP^T
        float st[8][4], dpt[8][4];
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) { st[j][e] = 0.f; dpt[j][e] = 0.f; }
        am_mm_rows(st, ka, Qs[buf]);
        am_mm_rows(dpt, va, dOs[buf]);
        const bool diag = q0 < wk0 + 15;
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int qi = j * 8 + 2 * t + (e & 1);             // query within the block
                const int key = wk0 + g + (e >> 1) * 8;
                float p = exp2f(st[j][e] * sl2 - Lq[j][e & 1]);
                if ((diag && key > q0 + qi) || q0 + qi >= Tn) p = 0.f;
                st[j][e] = p;                                        // P^T
                dpt[j][e] = p * (dpt[j][e] - Dq[j][e & 1]);          // dS^T
            }
        uint32_t pa[4][4], dsa[4][4];
        am_acc_to_afrag(pa, st);
        am_acc_to_afrag(dsa, dpt);
        am_mm_cols(dv, pa, dOs[buf]);
        am_mm_cols(dk, dsa, Qs[buf]);
    }
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int key = wk0 + g + r * 8;
        if (key >= Tn) continue;
        bf16* row = dqkv + ((size_t)b * Tn + key) * C3 + h * AM_HS;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            *reinterpret_cast<uint32_t*>(row + C + j * 8 + 2 * t) =
                am_pack(dk[j][2 * r] * 0.125f, dk[j][2 * r + 1] * 0.125f);
            *reinterpret_cast<uint32_t*>(row + 2 * C + j * 8 + 2 * t) = am_pack(dv[j][2 * r], dv[j][2 * r + 1]);
        }
    }
}

// ============================================================== backward: dQ
__global__ void __launch_bounds__(AMB_THREADS)
attention_backward_dq_mma(bf16* __restrict__ dqkv, const bf16* __restrict__ dout, const bf16* __restrict__ qkv,
                          const float* __restrict__ lse, const float* __restrict__ Dsum, int B, int Tn, int C,
                          int NH) {
    __shared__ __align__(128) bf16 Qs[AMB_ROWS * AM_HS];
    __shared__ __align__(128) bf16 dOs[AMB_ROWS * AM_HS];
    __shared__ __align__(128) bf16 Ks[2][AMB_ROWS * AM_HS];
    __shared__ __align__(128) bf16 Vs[2][AMB_ROWS * AM_HS];
    const int nb = (Tn + AMB_ROWS - 1) / AMB_ROWS;
    const int qbi = nb - 1 - blockIdx.x;          // longest rows first
    const int bh = blockIdx.y, b = bh / NH, h = bh % NH;
    const int C3 = 3 * C;
    const bf16* base = qkv + (size_t)b * Tn * C3;
    const bf16* qg = base + h * AM_HS;
    const bf16* kg = base + C + h * AM_HS;
    const bf16* vg = base + 2 * C + h * AM_HS;
    const bf16* dog = dout + (size_t)b * Tn * C + h * AM_HS;
    const int warp = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
    const int q0 = qbi * AMB_ROWS;
    const int wq0 = q0 + warp * 16;

    am_load_tile<AMB_ROWS, AMB_THREADS>(Qs, qg, C3, q0, Tn);
    am_load_tile<AMB_ROWS, AMB_THREADS>(dOs, dog, C, q0, Tn);
    am_load_tile<AMB_ROWS, AMB_THREADS>(Ks[0], kg, C3, 0, Tn);
    am_load_tile<AMB_ROWS, AMB_THREADS>(Vs[0], vg, C3, 0, Tn);
    am_cp_commit();

    float Lr[2], Dr[2];
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int q = wq0 + g + r * 8;
        Lr[r] = q < Tn ? lse[(size_t)bh * Tn + q] * AM_LOG2E : 0.f;
        Dr[r] = q < Tn ? Dsum[(size_t)bh * Tn + q] : 0.f;
    }
    const float sl2 = AM_LOG2E / 8.0f;
    uint32_t qa[4][4], doa[4][4];
    float dq[8][4];
#pragma unroll
    for (int j = 0; j < 8; j++) dq[j][0] = dq[j][1] = dq[j][2] = dq[j][3] = 0.f;

    for (int kb = 0; kb <= qbi; kb++) {
        const int buf = kb & 1;
        if (kb + 1 <= qbi) {
            __syncthreads();
            am_load_tile<AMB_ROWS, AMB_THREADS>(Ks[buf ^ 1], kg, C3, (kb + 1) * AMB_ROWS, Tn);
            am_load_tile<AMB_ROWS, AMB_THREADS>(Vs[buf ^ 1], vg, C3, (kb + 1) * AMB_ROWS, Tn);
        }
        am_cp_commit();
        am_cp_wait<1>();
        __syncthreads();
        if (kb == 0) {
            am_load_afrag(qa, Qs, warp * 16);
            am_load_afrag(doa, dOs, warp * 16);
        }
        const int k0 = kb * AMB_ROWS;
        if (k0 > wq0 + 15) continue;               // every key of the block follows this warp's queries
        float s[8][4], dp[8][4];
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) { s[j][e] = 0.f; dp[j][e] = 0.f; }
        am_mm_rows(s, qa, Ks[buf]);
        am_mm_rows(dp, doa, Vs[buf]);
        const bool diag = k0 + AMB_ROWS - 1 > wq0;
#pragma unroll
        for (int j = 0; j < 8; j++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int key = k0 + j * 8 + 2 * t + (e & 1);
                const int r = e >> 1;
                const int q = wq0 + g + r * 8;
                float p = exp2f(s[j][e] * sl2 - Lr[r]);
                if (diag && key > q) p = 0.f;
                s[j][e] = p * (dp[j][e] - Dr[r]);                    // dS
            }
        uint32_t dsa[4][4];
        am_acc_to_afrag(dsa, s);
        am_mm_cols(dq, dsa, Ks[buf]);
    }
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int q = wq0 + g + r * 8;
        if (q >= Tn) continue;
        bf16* row = dqkv + ((size_t)b * Tn + q) * C3 + h * AM_HS;
#pragma unroll
        for (int j = 0; j < 8; j++)
            *reinterpret_cast<uint32_t*>(row + j * 8 + 2 * t) = am_pack(dq[j][2 * r] * 0.125f, dq[j][2 * r + 1] * 0.125f);
    }
}
